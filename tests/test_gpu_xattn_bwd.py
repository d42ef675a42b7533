"""GPU parity of the output copies' gradient (orthros_xattn_bwd: Eq. (5) with the
copies' scale-offset) against the fp64 oracle's xattn_bwd, and of a whole training
step's attention gradient (orthros_swa_bwd, then orthros_xattn_bwd adding the
copies' share into dK / dV) against the sum of the two oracle gradients.  The bar
is the one of the base-stream gradient tests (normwise 1e-2, elementwise 3e-2 of
the tensor's largest magnitude), derived there from the bf16 operand roundings."""
import math

import numpy as np
import pytest
import torch

import long_context_attention_orthros_gb300 as orth
import oracle
from synthetic import normal_bf16, scale_offset
from tests.gpu_util import bf, dev, f32, i32
from tests.test_gpu_swa_bwd import NAMES, _assert_grad, _inputs

pytestmark = pytest.mark.gpu


def _copies(seed, B, T_kv, T_out, Hq, d, positions):
    qc = normal_bf16(seed, "qc_raw", (B, T_out, Hq, d))
    dOc = normal_bf16(seed, "dOc", (B, T_out, Hq, d))
    ac, bc = scale_offset(seed, Hq, d, prefix="_c")
    g = np.random.default_rng(seed)
    if positions == "every":
        pos = np.tile(np.arange(T_out, dtype=np.int32), (B, 1))
    elif positions == "tail_shuffled":
        pos = np.stack([g.permutation(np.arange(T_kv - T_out, T_kv)) for _ in range(B)]).astype(np.int32)
    else:  # random with duplicates, first and last position present
        pos = g.integers(0, T_kv, size=(B, T_out)).astype(np.int32)
        pos[:, 0] = T_kv - 1
        if T_out > 1:
            pos[:, 1] = 0
        if T_out > 3:
            pos[:, 3] = pos[:, 2]
    return qc, pos, dOc, ac, bc


def _gpu_xattn_grads(qc, pos, k, v, ac, bc, dOc, scale, dk=None, dv=None):
    qg, kg, vg, dOg, pg = bf(qc), bf(k), bf(v), bf(dOc), i32(pos)
    ag, bg = f32(ac), f32(bc)
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    oc = orth.xattn_fwd(qg, pg, kg, vg, ag, bg, scale=scale)
    got = orth.xattn_bwd(qg, pg, kg, vg, ag, bg, oc, dOg, scale=scale, dk=dk, dv=dv, dev_err=err)
    torch.cuda.synchronize()
    return [t.cpu().numpy().astype(np.float64) for t in got], int(err.item())


@pytest.mark.parametrize("B,T_kv,T_out,Hq,Hkv,d,positions", [
    (2, 300, 20, 8, 2, 128, "random"),         # duplicates, positions 0 and T_kv-1
    (1, 500, 64, 32, 8, 128, "tail_shuffled"),  # SFT layout at reduced size
    (1, 200, 7, 4, 4, 64, "random"),           # G=1, d=64
    (1, 130, 130, 8, 1, 64, "every"),          # PT mode: a copy at every position, G=8
    (2, 100, 1, 32, 8, 128, "tail_shuffled"),  # one copy at the last position (inference layout)
    (1, 77, 5, 16, 1, 128, "random"),          # G=16, ragged key tail
])
def test_xattn_bwd_parity(B, T_kv, T_out, Hq, Hkv, d, positions):
    seed = 5000 + T_kv + T_out
    _, k, v, _, _, _ = _inputs(seed, B, T_kv, Hq, Hkv, d)
    qc, pos, dOc, ac, bc = _copies(seed, B, T_kv, T_out, Hq, d, positions)
    scale = 1.0 / math.sqrt(d)
    got, err = _gpu_xattn_grads(qc, pos, k, v, ac, bc, dOc, scale)
    assert err == 0
    ref = oracle.xattn_bwd(qc, pos, k, v, ac, bc, dOc, scale)
    for name, g, r in zip(NAMES, got, ref):
        _assert_grad(g, r, name)


def test_training_step_gradient_adds_the_copies_share():
    """swa_bwd, then xattn_bwd with the same dK / dV buffers: the sum of both oracle
    gradients for K and V, each stream's own for its queries and scale-offset."""
    B, T, T_out, Hq, Hkv, d, w = 2, 400, 48, 16, 4, 128, 128
    q, k, v, a, b, dO = _inputs(6001, B, T, Hq, Hkv, d)
    qc, pos, dOc, ac, bc = _copies(6001, B, T, T_out, Hq, d, "tail_shuffled")
    scale = 1.0 / math.sqrt(d)
    qg, kg, vg, dOg, ag, bg = bf(q), bf(k), bf(v), bf(dO), f32(a), f32(b)
    o = orth.swa_fwd(qg, kg, vg, ag, bg, window=w, scale=scale)
    dq, dk, dv, da, db = orth.swa_bwd(qg, kg, vg, ag, bg, o, dOg, window=w, scale=scale)
    (dqc, dk2, dv2, dac, dbc), err = _gpu_xattn_grads(qc, pos, k, v, ac, bc, dOc, scale, dk=dk, dv=dv)
    assert err == 0
    rb = oracle.swa_bwd(q, k, v, a, b, dO, w, scale)
    rc = oracle.xattn_bwd(qc, pos, k, v, ac, bc, dOc, scale)
    _assert_grad(dq.cpu().numpy().astype(np.float64), rb[0], "dq_raw")
    _assert_grad(dk2, rb[1] + rc[1], "dk (base + copies)")
    _assert_grad(dv2, rb[2] + rc[2], "dv (base + copies)")
    _assert_grad(dqc, rc[0], "dqc_raw")
    _assert_grad(dac, rc[3], "dalpha_c")
    _assert_grad(dbc, rc[4], "dbeta_c")
    _assert_grad(da.cpu().numpy().astype(np.float64), rb[3], "dalpha")
    _assert_grad(db.cpu().numpy().astype(np.float64), rb[4], "dbeta")


def test_xattn_bwd_bad_position_gets_zeros_and_the_error_bit():
    B, T_kv, T_out, Hq, Hkv, d = 1, 150, 6, 8, 2, 128
    _, k, v, _, _, _ = _inputs(6100, B, T_kv, Hq, Hkv, d)
    qc, pos, dOc, ac, bc = _copies(6100, B, T_kv, T_out, Hq, d, "random")
    bad = pos.copy()
    bad[0, 2] = T_kv  # one past the last key
    scale = 1.0 / math.sqrt(d)
    (dq, dk, dv, da, db), err = _gpu_xattn_grads(qc, bad, k, v, ac, bc, dOc, scale)
    assert err & orth.DEVERR_POSITION
    assert not dq[0, 2].any()
    keep = [i for i in range(T_out) if i != 2]
    ref = oracle.xattn_bwd(np.ascontiguousarray(qc[:, keep]), np.ascontiguousarray(pos[:, keep]), k, v, ac, bc,
                           np.ascontiguousarray(dOc[:, keep]), scale)
    for name, g, r in zip(NAMES, (dq[:, keep], dk, dv, da, db), ref):
        _assert_grad(g, r, name)


def test_xattn_bwd_without_copies():
    """T_out = 0: dK / dV passed in stay as they are; fresh ones come back zero."""
    B, T_kv, Hq, Hkv, d = 1, 90, 8, 2, 64
    k = bf(normal_bf16(1, "k", (B, T_kv, Hkv, d)))
    v = bf(normal_bf16(1, "v", (B, T_kv, Hkv, d)))
    e = torch.empty((B, 0, Hq, d), dtype=torch.bfloat16, device=dev())
    pos = torch.empty((B, 0), dtype=torch.int32, device=dev())
    ac = torch.ones((Hq, d), dtype=torch.float32, device=dev())
    dk0 = torch.randn((B, T_kv, Hkv, d), device=dev())
    dv0 = torch.randn((B, T_kv, Hkv, d), device=dev())
    dk1, dv1 = dk0.clone(), dv0.clone()
    out = orth.xattn_bwd(e, pos, k, v, ac, ac, e, e, dk=dk1, dv=dv1)
    torch.cuda.synchronize()
    assert torch.equal(dk1, dk0) and torch.equal(dv1, dv0)
    assert out[0].numel() == 0 and not out[3].any() and not out[4].any()
    fresh = orth.xattn_bwd(e, pos, k, v, ac, ac, e, e)
    torch.cuda.synchronize()
    assert not fresh[1].any() and not fresh[2].any()


def test_xattn_bwd_sft_sized_copies():
    """A 16K-token sequence with 8B-class heads and 512 copies of positions among the
    last 2048 (shuffled): every output against the oracle."""
    B, T_kv, T_out, Hq, Hkv, d = 1, 16384, 512, 32, 8, 128
    seed = 6200
    _, k, v, _, _, _ = _inputs(seed, B, T_kv, Hq, Hkv, d)
    qc, _, dOc, ac, bc = _copies(seed, B, T_kv, T_out, Hq, d, "random")
    g = np.random.default_rng(seed)
    pos = g.permutation(np.arange(T_kv - 2048, T_kv))[:T_out].astype(np.int32).reshape(1, T_out)
    scale = 1.0 / math.sqrt(d)
    got, err = _gpu_xattn_grads(qc, pos, k, v, ac, bc, dOc, scale)
    assert err == 0
    ref = oracle.xattn_bwd(qc, pos, k, v, ac, bc, dOc, scale)
    for name, gg, r in zip(NAMES, got, ref):
        _assert_grad(gg, r, name)


@pytest.mark.parametrize("positions", [[16383, 5000, 0], [700, 20, 999]])
def test_xattn_bwd_few_copies_over_long_keys(positions):
    """A few copies over a 16K-token sequence (8B-class heads): their dq runs with the keys
    split over many CTAs (per-split max and sum, a combine, then per-split dq added up).
    The second case puts every copy early, so most splits see no key at all."""
    B, T_kv, Hq, Hkv, d = 1, 16384, 32, 8, 128
    T_out = len(positions)
    seed = 6300 + positions[0]
    _, k, v, _, _, _ = _inputs(seed, B, T_kv, Hq, Hkv, d)
    qc, _, dOc, ac, bc = _copies(seed, B, T_kv, T_out, Hq, d, "random")
    pos = np.array([positions], np.int32)
    scale = 1.0 / math.sqrt(d)
    got, err = _gpu_xattn_grads(qc, pos, k, v, ac, bc, dOc, scale)
    assert err == 0
    ref = oracle.xattn_bwd(qc, pos, k, v, ac, bc, dOc, scale)
    for name, g, r in zip(NAMES, got, ref):
        _assert_grad(g, r, name)
