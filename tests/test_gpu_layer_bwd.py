"""GPU parity of a layer's whole attention gradient in one call (orthros_attn_bwd: the base
stream's Eq. (4) and the output copies' Eq. (5), each with its scale-offset, dK / dV holding
both shares) against the fp64 oracle: swa_bwd of the base stream plus xattn_bwd of the copies.
The bar is the one of the single-stream gradient tests (normwise 1e-2, elementwise 3e-2 of the
tensor's largest magnitude), derived there from the bf16 operand roundings."""
import math

import numpy as np
import pytest
import torch

import long_context_attention_orthros_gb300 as orth
import oracle
from tests.gpu_util import bf, dev, f32, i32
from tests.test_gpu_swa_bwd import _assert_grad, _inputs
from tests.test_gpu_xattn_bwd import _copies

pytestmark = pytest.mark.gpu

LAYER_NAMES = ("dq_raw", "dk", "dv", "dalpha", "dbeta", "dqc_raw", "dalpha_c", "dbeta_c")


def _layer(seed, B, T, T_out, Hq, Hkv, d, w, positions, with_lse, pos_override=None):
    q, k, v, a, b, dO = _inputs(seed, B, T, Hq, Hkv, d)
    qc, pos, dOc, ac, bc = _copies(seed, B, T, T_out, Hq, d, positions)
    if pos_override is not None:
        pos = pos_override
    scale = 1.0 / math.sqrt(d)
    qg, kg, vg, ag, bg = bf(q), bf(k), bf(v), f32(a), f32(b)
    qcg, pg, acg, bcg = bf(qc), i32(pos), f32(ac), f32(bc)
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    if with_lse:
        o, lse = orth.swa_fwd_lse(qg, kg, vg, ag, bg, window=w, scale=scale)
        oc, lsec = orth.xattn_fwd(qcg, pg, kg, vg, acg, bcg, scale=scale, lse=True, dev_err=err)
    else:
        o = orth.swa_fwd(qg, kg, vg, ag, bg, window=w, scale=scale)
        oc = orth.xattn_fwd(qcg, pg, kg, vg, acg, bcg, scale=scale, dev_err=err)
        lse = lsec = None
    got = orth.attn_bwd(qg, kg, vg, ag, bg, o, bf(dO), qcg, pg, acg, bcg, oc, bf(dOc), window=w, scale=scale,
                        lse=lse, lsec=lsec, dev_err=err)
    torch.cuda.synchronize()
    got = [t.cpu().numpy().astype(np.float64) for t in got]
    return got, int(err.item()), (q, k, v, a, b, dO, qc, pos, dOc, ac, bc, scale)


def _reference(inp, w):
    q, k, v, a, b, dO, qc, pos, dOc, ac, bc, scale = inp
    rb = oracle.swa_bwd(q, k, v, a, b, dO, w, scale)
    rc = oracle.xattn_bwd(qc, pos, k, v, ac, bc, dOc, scale)
    return (rb[0], rb[1] + rc[1], rb[2] + rc[2], rb[3], rb[4], rc[0], rc[3], rc[4])


@pytest.mark.parametrize("B,T,T_out,Hq,Hkv,d,w,positions,with_lse", [
    (2, 400, 48, 16, 4, 128, 128, "tail_shuffled", True),   # SFT layout at reduced size
    (2, 400, 48, 16, 4, 128, 128, "tail_shuffled", False),  # without the forwards' log-sum-exp
    (2, 3000, 1, 32, 8, 128, 128, "tail_shuffled", True),   # one copy per sequence: the split copy dq
    (1, 3000, 3, 32, 8, 128, 128, "random", False),         # few copies, no lse: split dq, both passes
    (1, 130, 130, 8, 1, 64, 128, "every", True),            # PT mode: a copy at every position, G=8
    (1, 300, 20, 8, 2, 128, 33, "random", True),            # duplicates, positions 0 and T-1, narrow window
    (1, 700, 300, 32, 8, 128, 128, "random", True),         # many copies (tensor-memory forward), ragged tails
])
def test_layer_gradient_matches_both_oracle_streams(B, T, T_out, Hq, Hkv, d, w, positions, with_lse):
    got, err, inp = _layer(9000 + T + T_out, B, T, T_out, Hq, Hkv, d, w, positions, with_lse)
    assert err == 0
    for name, g, r in zip(LAYER_NAMES, got, _reference(inp, w)):
        _assert_grad(g, r, name)


def test_layer_gradient_without_copies_is_the_base_gradient():
    B, T, Hq, Hkv, d, w = 1, 500, 8, 2, 128, 128
    got, err, inp = _layer(9100, B, T, 0, Hq, Hkv, d, w, "every", True)
    assert err == 0
    q, k, v, a, b, dO = inp[:6]
    rb = oracle.swa_bwd(q, k, v, a, b, dO, w, inp[-1])
    for name, g, r in zip(LAYER_NAMES[:5], got[:5], rb):
        _assert_grad(g, r, name)
    assert got[5].size == 0 and not got[6].any() and not got[7].any()


def test_layer_gradient_equals_the_two_calls():
    """The one-call gradient against swa_bwd then xattn_bwd (accumulating) on the GPU: the same
    roundings, so the results agree to fp32 summation order."""
    B, T, T_out, Hq, Hkv, d, w = 2, 600, 64, 32, 8, 128, 128
    q, k, v, a, b, dO = _inputs(9200, B, T, Hq, Hkv, d)
    qc, pos, dOc, ac, bc = _copies(9200, B, T, T_out, Hq, d, "tail_shuffled")
    qg, kg, vg, ag, bg = bf(q), bf(k), bf(v), f32(a), f32(b)
    qcg, pg, acg, bcg = bf(qc), i32(pos), f32(ac), f32(bc)
    o, lse = orth.swa_fwd_lse(qg, kg, vg, ag, bg, window=w)
    oc, lsec = orth.xattn_fwd(qcg, pg, kg, vg, acg, bcg, lse=True)
    one = orth.attn_bwd(qg, kg, vg, ag, bg, o, bf(dO), qcg, pg, acg, bcg, oc, bf(dOc), window=w, lse=lse,
                        lsec=lsec)
    base = orth.swa_bwd(qg, kg, vg, ag, bg, o, bf(dO), window=w, lse=lse)
    copy = orth.xattn_bwd(qcg, pg, kg, vg, acg, bcg, oc, bf(dOc), dk=base[1], dv=base[2], lse=lsec)
    torch.cuda.synchronize()
    two = (base[0], copy[1], copy[2], base[3], base[4], copy[0], copy[3], copy[4])
    for name, x, y in zip(LAYER_NAMES, one, two):
        x, y = x.double(), y.double()
        assert float((x - y).norm()) <= 1e-5 * float(y.norm()), name


def test_layer_gradient_bad_position_gets_zeros_and_the_error_bit():
    B, T, T_out, Hq, Hkv, d, w = 1, 300, 8, 8, 2, 128, 128
    g = np.random.default_rng(1)
    pos = g.integers(0, T, size=(B, T_out)).astype(np.int32)
    bad = pos.copy()
    bad[0, 3] = T  # one past the last key
    got, err, inp = _layer(9300, B, T, T_out, Hq, Hkv, d, w, "random", False, pos_override=bad)
    assert err & orth.DEVERR_POSITION
    assert not got[5][0, 3].any()
    keep = [i for i in range(T_out) if i != 3]
    q, k, v, a, b, dO, qc, _, dOc, ac, bc, scale = inp
    ref = _reference((q, k, v, a, b, dO, np.ascontiguousarray(qc[:, keep]), np.ascontiguousarray(pos[:, keep]),
                      np.ascontiguousarray(dOc[:, keep]), ac, bc, scale), w)
    got[5] = got[5][:, keep]
    for name, gg, r in zip(LAYER_NAMES, got, ref):
        _assert_grad(gg, r, name)
