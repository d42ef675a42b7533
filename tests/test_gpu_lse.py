"""GPU parity of the forward's per-row log-sum-exp (orthros_swa_fwd_lse for the base stream,
orthros_xattn_fwd_lse for the output copies) against the fp64 oracle, and of the gradients that
take it (orthros_swa_bwd with lse: the persistent tensor-memory dq kernel; orthros_xattn_bwd
with lse: the copies' dq in one pass) against the oracle's gradients.

Bar for lse: 1e-2 absolute.  The kernels take q . k with q rounded once to fp16 (tensor-memory
path) or as a bf16 high part plus residual (warp path), i.e. each logit within ~2^-11 of its
size (|scale q . k| <= ~11 for these N(0,1) inputs: <= ~5e-3), and a log-sum-exp moves by no
more than its largest logit does."""
import math

import numpy as np
import pytest
import torch

import long_context_attention_orthros_gb300 as orth
import oracle
from synthetic import normal_bf16, scale_offset
from tests.gpu_util import bf, dev, f32
from tests.test_gpu_swa_bwd import NAMES, _assert_grad, _inputs

pytestmark = pytest.mark.gpu

LSE_ABS = 1e-2


@pytest.mark.parametrize("B,T,Hq,Hkv,d,w", [
    (2, 1000, 32, 8, 128, 128),   # tensor-memory path, ragged tail
    (1, 300, 8, 2, 64, 128),      # d=64
    (1, 257, 16, 1, 128, 33),     # G=16, narrow window
    (1, 640, 8, 2, 128, 600),     # band too wide for tensor memory: warp path
    (1, 5, 4, 1, 128, 128),       # T smaller than a tile
])
def test_forward_lse_matches_oracle(B, T, Hq, Hkv, d, w):
    q = normal_bf16(7000 + T, "q_raw", (B, T, Hq, d))
    k = normal_bf16(7000 + T, "k", (B, T, Hkv, d))
    v = normal_bf16(7000 + T, "v", (B, T, Hkv, d))
    a, b = scale_offset(7000 + T, Hq, d)
    scale = 1.0 / math.sqrt(d)
    qg, kg, vg, ag, bg = bf(q), bf(k), bf(v), f32(a), f32(b)
    o, lse = orth.swa_fwd_lse(qg, kg, vg, ag, bg, window=w, scale=scale)
    o_plain = orth.swa_fwd(qg, kg, vg, ag, bg, window=w, scale=scale)
    torch.cuda.synchronize()
    assert torch.equal(o, o_plain)  # asking for lse changes nothing else
    got = lse.cpu().numpy().astype(np.float64)
    ref = oracle.swa_lse(q, k, a, b, w, scale)
    err = float(np.abs(got - ref).max())
    assert err <= LSE_ABS, f"lse max |err| {err:.3e}"


@pytest.mark.parametrize("B,T,Hq,Hkv,d,w", [
    (1, 300, 8, 2, 128, 128),
    (2, 257, 16, 2, 128, 128),
    (1, 640, 8, 2, 128, 600),
    (2, 4000, 16, 4, 128, 128),  # 1000 row tiles: each persistent CTA walks several
    (1, 3000, 32, 8, 64, 128),   # d=64, 752 row tiles, ragged last tile
    (1, 1000, 16, 1, 128, 128),  # G=16: band dq, dalpha / dbeta in their own pass
    (1, 700, 8, 2, 128, 129),    # G=4, the widest window whose band fits the key ring
    (1, 700, 8, 2, 128, 130),    # one key wider: 64-key blocks
    (1, 600, 4, 2, 128, 128),    # G=2: 64-key blocks
    (2, 333, 8, 1, 64, 50),      # G=8, d=64, narrow window
    (3, 2000, 8, 2, 128, 97),    # three sequences per KV head group over the CTAs' tile runs
])
def test_gradient_with_forward_lse(B, T, Hq, Hkv, d, w):
    q, k, v, a, b, dO = _inputs(3000 + T, B, T, Hq, Hkv, d)
    scale = 1.0 / math.sqrt(d)
    qg, kg, vg, dOg, ag, bg = bf(q), bf(k), bf(v), bf(dO), f32(a), f32(b)
    o, lse = orth.swa_fwd_lse(qg, kg, vg, ag, bg, window=w, scale=scale)
    got = orth.swa_bwd(qg, kg, vg, ag, bg, o, dOg, window=w, scale=scale, lse=lse)
    torch.cuda.synchronize()
    ref = oracle.swa_bwd(q, k, v, a, b, dO, w, scale)
    for name, g, r in zip(NAMES, got, ref):
        _assert_grad(g.cpu().numpy().astype(np.float64), r, name)


def test_gradient_full_size_sampled():
    """The bench's gradient at its full size (2 x 131072 tokens, 32/8 heads, d=128, w=128, one
    copy per sequence at its last position), launched as bench.py launches it: forwards with
    their log-sum-exp, then both streams' gradient in one call (orthros_attn_bwd).
    Sampled base rows and keys against the oracle on the slices they depend on (a base row
    on the w tokens up to it, a key on the tokens j-w+1..j+w-1), the copy's share of those
    keys from the oracle's copy gradient, every copy row in full, and dalpha / dbeta as the
    sums they are over the GPU's own dq."""
    from tests.test_gpu_swa_bwd import _slice_grads
    from tests.gpu_util import i32
    B, T, Hq, Hkv, d, w = 2, 131072, 32, 8, 128, 128
    q, k, v, a, b, dO = _inputs(8800, B, T, Hq, Hkv, d)
    qc = normal_bf16(8800, "qc_raw", (B, 1, Hq, d))
    dOc = normal_bf16(8800, "dOc", (B, 1, Hq, d))
    ac, bc = scale_offset(8800, Hq, d, prefix="_c")
    pos = np.full((B, 1), T - 1, np.int32)
    scale = 1.0 / math.sqrt(d)
    qg, kg, vg, ag, bg = bf(q), bf(k), bf(v), f32(a), f32(b)
    o, lse = orth.swa_fwd_lse(qg, kg, vg, ag, bg, window=w, scale=scale)
    qcg, pg = bf(qc), i32(pos)
    oc, lsec = orth.xattn_fwd(qcg, pg, kg, vg, f32(ac), f32(bc), scale=scale, lse=True)
    dq, dk, dv, da, db, dqc, dac, dbc = orth.attn_bwd(qg, kg, vg, ag, bg, o, bf(dO), qcg, pg, f32(ac), f32(bc), oc,
                                                      bf(dOc), window=w, scale=scale, lse=lse, lsec=lsec)
    torch.cuda.synchronize()
    del o, oc, lse, lsec
    rc = oracle.xattn_bwd(qc, pos, k, v, ac, bc, dOc, scale)  # the copy's share, every key
    for name, g, r in zip(("dqc_raw", "dalpha_c", "dbeta_c"), (dqc, dac, dbc), (rc[0], rc[3], rc[4])):
        _assert_grad(g.cpu().numpy().astype(np.float64), r, name)
    for bb in range(B):
        for t in (0, 1, 127, 128, 65535, 65536, 99999, T - 2, T - 1):
            lo = max(0, t - w + 1)
            r = _slice_grads(q[bb:bb + 1], k[bb:bb + 1], v[bb:bb + 1], a, b, dO[bb:bb + 1], w, scale, lo, t + 1)
            _assert_grad(dq[bb, t].cpu().numpy().astype(np.float64), r[0][0, t - lo], f"dq_raw b{bb} row {t}")
        for j in (0, 63, 64, 777, 65536, 100000, T - 129, T - 65, T - 1):
            lo, hi = max(0, j - w + 1), min(T, j + w)
            r = _slice_grads(q[bb:bb + 1], k[bb:bb + 1], v[bb:bb + 1], a, b, dO[bb:bb + 1], w, scale, lo, hi)
            _assert_grad(dk[bb, j].cpu().numpy().astype(np.float64), r[1][0, j - lo] + rc[1][bb, j],
                         f"dk b{bb} key {j}")
            _assert_grad(dv[bb, j].cpu().numpy().astype(np.float64), r[2][0, j - lo] + rc[2][bb, j],
                         f"dv b{bb} key {j}")
    # the sums in float64 on the device (host copies of these would take tens of GB)
    dq_post = dq.double() / ag.double()  # dq = dq_raw / alpha
    db_ref = dq_post.sum(dim=(0, 1)).cpu().numpy()
    da_ref = (qg.double() * dq_post).sum(dim=(0, 1)).cpu().numpy()
    _assert_grad(db.cpu().numpy().astype(np.float64), db_ref, "dbeta as the sum of dq")
    _assert_grad(da.cpu().numpy().astype(np.float64), da_ref, "dalpha as the sum of x * dq")


def _copy_inputs(seed, B, T_kv, T_out, Hq, Hkv, d, positions):
    from tests.test_gpu_xattn_bwd import _copies
    _, k, v, _, _, _ = _inputs(seed, B, T_kv, Hq, Hkv, d)
    qc, pos, dOc, ac, bc = _copies(seed, B, T_kv, T_out, Hq, d, positions)
    return qc, pos, k, v, ac, bc, dOc


# (B, T_kv, T_out, Hq, Hkv, d, positions): which forward path writes the lse
XATTN_LSE_CASES = [
    (1, 2000, 256, 32, 8, 128, "tail_shuffled"),  # T_out * G >= 256: tensor-memory kernel
    (2, 300, 20, 8, 2, 128, "random"),           # split-KV partials and the combine
    (1, 200, 40, 8, 2, 64, "random"),            # one partial per row: written directly, d=64
    (2, 5000, 1, 32, 8, 128, "tail_shuffled"),   # one copy per sequence (the inference layout)
]


@pytest.mark.parametrize("B,T_kv,T_out,Hq,Hkv,d,positions", XATTN_LSE_CASES)
def test_copy_forward_lse_matches_oracle(B, T_kv, T_out, Hq, Hkv, d, positions):
    from tests.gpu_util import i32
    qc, pos, k, v, ac, bc, _ = _copy_inputs(7100 + T_kv + T_out, B, T_kv, T_out, Hq, Hkv, d, positions)
    scale = 1.0 / math.sqrt(d)
    args = (bf(qc), i32(pos), bf(k), bf(v), f32(ac), f32(bc))
    oc, lse = orth.xattn_fwd(*args, scale=scale, lse=True)
    oc_plain = orth.xattn_fwd(*args, scale=scale)
    torch.cuda.synchronize()
    assert torch.equal(oc, oc_plain)  # asking for lse changes nothing else
    got = lse.cpu().numpy().astype(np.float64)
    ref = oracle.xattn_lse(qc, pos, k, ac, bc, scale)
    err = float(np.abs(got - ref).max())
    assert err <= LSE_ABS, f"lse max |err| {err:.3e}"


def test_copy_forward_lse_of_a_bad_position_is_minus_infinity():
    from tests.gpu_util import i32
    B, T_kv, T_out, Hq, Hkv, d = 1, 300, 20, 8, 2, 128
    qc, pos, k, v, ac, bc, _ = _copy_inputs(7200, B, T_kv, T_out, Hq, Hkv, d, "random")
    bad = pos.copy()
    bad[0, 5] = T_kv
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    scale = 1.0 / math.sqrt(d)
    _, lse = orth.xattn_fwd(bf(qc), i32(bad), bf(k), bf(v), f32(ac), f32(bc), scale=scale, lse=True, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & orth.DEVERR_POSITION
    got = lse.cpu().numpy().astype(np.float64)
    assert np.all(np.isneginf(got[0, 5]))
    keep = [i for i in range(T_out) if i != 5]
    ref = oracle.xattn_lse(np.ascontiguousarray(qc[:, keep]), np.ascontiguousarray(pos[:, keep]), k, ac, bc, scale)
    assert float(np.abs(got[:, keep] - ref).max()) <= LSE_ABS


@pytest.mark.parametrize("B,T_kv,T_out,Hq,Hkv,d,positions", XATTN_LSE_CASES + [
    (1, 16384, 3, 32, 8, 128, "random"),  # few copies over long keys: the split dq, second pass only
    # at most 8 copy rows per KV head: the warp-MMA dq with the rows on N
    (1, 100, 1, 32, 8, 128, "tail_shuffled"),  # one split: dq stored, not added
    (2, 16384, 2, 8, 4, 128, "random"),        # G=2, positions anywhere (0 included)
    (1, 3000, 1, 16, 2, 64, "random"),         # G=8, d=64
    (1, 5000, 8, 4, 4, 128, "random"),         # G=1, 8 copies
    (3, 20000, 2, 32, 8, 128, "tail_shuffled"),  # 8 rows, 3 sequences, keys off the block grid
])
def test_copy_gradient_with_forward_lse(B, T_kv, T_out, Hq, Hkv, d, positions):
    from tests.gpu_util import i32
    qc, pos, k, v, ac, bc, dOc = _copy_inputs(7300 + T_kv + T_out, B, T_kv, T_out, Hq, Hkv, d, positions)
    scale = 1.0 / math.sqrt(d)
    args = (bf(qc), i32(pos), bf(k), bf(v), f32(ac), f32(bc))
    oc, lse = orth.xattn_fwd(*args, scale=scale, lse=True)
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    got = orth.xattn_bwd(*args, oc, bf(dOc), scale=scale, lse=lse, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.xattn_bwd(qc, pos, k, v, ac, bc, dOc, scale)
    for name, g, r in zip(NAMES, got, ref):
        _assert_grad(g.cpu().numpy().astype(np.float64), r, name)


def test_copy_gradient_with_forward_lse_bad_positions_few_rows():
    """The warp-MMA copies' dq (at most 8 rows per KV head): a copy with a position outside the
    keys gets a zero dq row, adds nothing to dalpha / dbeta, and sets the position bit."""
    from tests.gpu_util import i32
    B, T_kv, T_out, Hq, Hkv, d = 2, 9000, 2, 32, 8, 128
    qc, pos, k, v, ac, bc, dOc = _copy_inputs(7400, B, T_kv, T_out, Hq, Hkv, d, "random")
    bad = pos.copy()
    bad[0, 1] = T_kv
    bad[1, 0] = -3
    scale = 1.0 / math.sqrt(d)
    args = (bf(qc), i32(bad), bf(k), bf(v), f32(ac), f32(bc))
    oc, lse = orth.xattn_fwd(*args, scale=scale, lse=True)
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    got = orth.xattn_bwd(*args, oc, bf(dOc), scale=scale, lse=lse, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & orth.DEVERR_POSITION
    dq = got[0].cpu().numpy().astype(np.float64)
    assert (dq[0, 1] == 0).all() and (dq[1, 0] == 0).all()
    # the valid copies alone, one sequence at a time, against the oracle
    ref0 = oracle.xattn_bwd(qc[:1, :1], pos[:1, :1], k[:1], v[:1], ac, bc, dOc[:1, :1], scale)
    ref1 = oracle.xattn_bwd(qc[1:, 1:], pos[1:, 1:], k[1:], v[1:], ac, bc, dOc[1:, 1:], scale)
    _assert_grad(dq[:1, :1], ref0[0], "dq of the valid copy, sequence 0")
    _assert_grad(dq[1:, 1:], ref1[0], "dq of the valid copy, sequence 1")
    for i, name in ((3, "dalpha"), (4, "dbeta")):
        _assert_grad(got[i].cpu().numpy().astype(np.float64), ref0[i] + ref1[i], name)
