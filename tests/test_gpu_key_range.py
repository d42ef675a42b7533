"""Keys outside fp16's range.  The tensor-memory kernels take q . k in fp16; a key row whose
largest |k| reaches 65520 is scaled into range by an exact power of two and its logits are
scaled back in fp32, so every finite bf16 key is an input of Eqs. (4)-(5) like any other.
Each case is checked against the fp64 oracle, with the device error word left at zero:

* whole key rows times 2^17 (huge logits: the softmax of the rows that see them saturates);
* key rows with one element at 2^17 whose partner column of q is tiny (moderate logits: the
  other elements of the shifted rows, scaled by 2^-3 in fp16, still decide the result);
* an infinite key sets ORTHROS_DEVERR_RANGE (no finite logit exists for it).
"""
import numpy as np
import pytest
import torch

import long_context_attention_orthros_gb300 as orth
import oracle
from synthetic import PrefillConfig, bf16_bits, bf16_to_f32, make_prefill
from tests.gpu_util import assert_parity, bf, dev, f32, i32, val

pytestmark = pytest.mark.gpu

BIG = 2.0 ** 17


def _inputs(cfg, seed, mode, one_positive=False):
    inp = make_prefill(cfg, seed)
    g = np.random.default_rng(seed)
    if mode == "rows":
        # whole key rows scaled to +-2^17 |k| (exact in bf16), 300 rows apart so that a window
        # holds at most one; with q >= 0 (|q_raw|, beta >= 0) their logits are decisively huge
        # (about 1e6 in log2 units): +: the softmax sits on that key, -: it ignores it.  Near-ties
        # between huge logits are left out on purpose: no fp32 logit resolves them
        rows = np.arange(37, cfg.T, 300)
        sign = np.where(np.arange(rows.size) % 2 == 0, 1.0, -1.0).astype(np.float32)
        if one_positive:  # copies see every row: one positive at most, the rest negative
            sign[:] = -1.0
            sign[rows.size // 2] = 1.0
        k = bf16_to_f32(inp.k)
        k[:, rows] = np.abs(k[:, rows]) * (sign[None, :, None, None] * np.float32(BIG))
        inp.k[...] = bf16_bits(k)
        inp.q_raw[...] = inp.q_raw & np.uint16(0x7FFF)
        inp.qc_raw[...] = inp.qc_raw & np.uint16(0x7FFF)
        inp.beta[...] = np.abs(inp.beta)
        inp.beta_c[...] = np.abs(inp.beta_c)
        inp.alpha[...] = np.abs(inp.alpha)
        inp.alpha_c[...] = np.abs(inp.alpha_c)
    else:  # one element per shifted row at 2^17; q's partner column tiny, beta's zero there
        rows = np.sort(g.choice(cfg.T, size=max(4, cfg.T // 97), replace=False))
        c = 5
        inp.k[:, rows, :, c] = bf16_bits(np.full(1, BIG, np.float32))[0]
        q = bf16_to_f32(inp.q_raw)
        q[..., c] *= np.float32(2.0 ** -20)
        inp.q_raw[...] = bf16_bits(q)
        inp.beta[:, c] = 0.0
        inp.beta_c[:, c] = 0.0
        if not cfg.appended:
            qc = bf16_to_f32(inp.qc_raw)
            qc[..., c] *= np.float32(2.0 ** -20)
            inp.qc_raw[...] = bf16_bits(qc)
    return inp


@pytest.mark.parametrize("mode", ["rows", "element"])
@pytest.mark.parametrize("Hq,Hkv,d", [(8, 2, 128), (4, 2, 64), (16, 1, 128), (4, 4, 128)])
def test_swa_takes_keys_beyond_fp16(mode, Hq, Hkv, d):
    cfg = PrefillConfig("big_k", B=2, T=1000, Hq=Hq, Hkv=Hkv, d=d)
    inp = _inputs(cfg, 71 + d + Hq, mode)
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    o = orth.swa_fwd(bf(inp.q_raw), bf(inp.k), bf(inp.v), f32(inp.alpha), f32(inp.beta), window=cfg.window,
                     scale=cfg.scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.swa(inp.q_raw, inp.k, inp.v, inp.alpha, inp.beta, cfg.window, cfg.scale)
    assert_parity(val(o), ref, f"swa with keys beyond fp16 ({mode})")


@pytest.mark.parametrize("mode", ["rows", "element"])
@pytest.mark.parametrize("T_out,Hq,Hkv,d", [(1, 32, 8, 128), (64, 8, 2, 128), (160, 4, 2, 64)])
def test_xattn_takes_keys_beyond_fp16(mode, T_out, Hq, Hkv, d):
    cfg = PrefillConfig("big_kc", B=2, T=3000, Hq=Hq, Hkv=Hkv, d=d, T_out=T_out, positions="shuffled")
    inp = _inputs(cfg, 91 + T_out + d, mode, one_positive=True)
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    oc = orth.xattn_fwd(bf(inp.qc_raw), i32(inp.pos), bf(inp.k), bf(inp.v), f32(inp.alpha_c), f32(inp.beta_c),
                        scale=cfg.scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.xattn(inp.qc_raw, inp.pos, inp.k, inp.v, inp.alpha_c, inp.beta_c, cfg.scale)
    assert_parity(val(oc), ref, f"xattn with keys beyond fp16 ({mode})")


@pytest.mark.parametrize("T_out", [1, 64])
def test_infinite_key_sets_the_range_flag(T_out):
    cfg = PrefillConfig("inf_k", B=1, T=600, Hq=8, Hkv=2, d=128, T_out=T_out)
    inp = make_prefill(cfg, 5)
    inp.k[0, 300, 1, 7] = 0x7F80  # +inf
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    k, v = bf(inp.k), bf(inp.v)
    orth.swa_fwd(bf(inp.q_raw), k, v, f32(inp.alpha), f32(inp.beta), scale=cfg.scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & orth.DEVERR_RANGE
    if T_out > 1:  # the tensor-memory copies kernel
        err.zero_()
        orth.xattn_fwd(bf(inp.qc_raw), i32(inp.pos), k, v, f32(inp.alpha_c), f32(inp.beta_c), scale=cfg.scale,
                       dev_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) & orth.DEVERR_RANGE


@pytest.mark.parametrize("mode", ["rows", "element"])
@pytest.mark.parametrize("T_out,Hq,Hkv,d", [(1, 32, 8, 128), (2, 8, 2, 64), (1, 16, 2, 128)])
def test_prefill_call_takes_keys_beyond_fp16(mode, T_out, Hq, Hkv, d):
    """One prefill layer through orthros_prefill_fwd with keys beyond fp16."""
    cfg = PrefillConfig("big_kp", B=2, T=2000, Hq=Hq, Hkv=Hkv, d=d, T_out=T_out)
    inp = _inputs(cfg, 131 + T_out + d, mode, one_positive=True)
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    o, oc = orth.prefill_fwd(bf(inp.q_raw), bf(inp.k), bf(inp.v), f32(inp.alpha), f32(inp.beta), bf(inp.qc_raw),
                             i32(inp.pos), f32(inp.alpha_c), f32(inp.beta_c), scale=cfg.scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.swa(inp.q_raw, inp.k, inp.v, inp.alpha, inp.beta, cfg.window, cfg.scale)
    ref_c = oracle.xattn(inp.qc_raw, inp.pos, inp.k, inp.v, inp.alpha_c, inp.beta_c, cfg.scale)
    assert_parity(val(o), ref, f"prefill call base with keys beyond fp16 ({mode})")
    assert_parity(val(oc), ref_c, f"prefill call copies with keys beyond fp16 ({mode})")


@pytest.mark.parametrize("B,T,T_out,Hq,Hkv,d,with_lse", [
    (2, 900, 40, 16, 4, 128, True),    # SFT-like layout: tensor-memory dq of the copies, persistent base dq
    (2, 900, 40, 16, 4, 128, False),   # without the forwards' log-sum-exp (two-pass copies dq)
    (1, 3000, 1, 32, 8, 128, True),    # one copy per sequence: the copies' dq split over the keys
    (1, 700, 30, 8, 2, 64, True),      # d = 64
])
def test_layer_gradient_takes_keys_beyond_fp16(B, T, T_out, Hq, Hkv, d, with_lse):
    """orthros_attn_bwd with key rows holding an element at 2^17 (moderate logits, as above): the
    gradient's fp16 copy of K is shifted per row, and every kernel reading q . k scales back.
    Same bar as the other gradient tests (normwise 1e-2, elementwise 3e-2 of the largest)."""
    import math
    from tests.test_gpu_layer_bwd import LAYER_NAMES, _reference
    from tests.test_gpu_swa_bwd import _assert_grad, _inputs
    from tests.test_gpu_xattn_bwd import _copies
    seed = 777 + T + T_out
    q, k, v, a, b, dO = _inputs(seed, B, T, Hq, Hkv, d)
    qc, pos, dOc, ac, bc = _copies(seed, B, T, T_out, Hq, d, "random")
    g = np.random.default_rng(seed)
    rows = np.sort(g.choice(T, size=max(4, T // 97), replace=False))
    c = 5
    k[:, rows, :, c] = bf16_bits(np.full(1, BIG, np.float32))[0]
    for x in (q, qc):
        xf = bf16_to_f32(x)
        xf[..., c] *= np.float32(2.0 ** -20)
        x[...] = bf16_bits(xf)
    b[:, c] = 0.0
    bc[:, c] = 0.0
    scale = 1.0 / math.sqrt(d)
    qg, kg, vg, ag, bg = bf(q), bf(k), bf(v), f32(a), f32(b)
    qcg, pg, acg, bcg = bf(qc), i32(pos), f32(ac), f32(bc)
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    if with_lse:
        o, lse = orth.swa_fwd_lse(qg, kg, vg, ag, bg, scale=scale, dev_err=err)
        oc, lsec = orth.xattn_fwd(qcg, pg, kg, vg, acg, bcg, scale=scale, lse=True, dev_err=err)
    else:
        o = orth.swa_fwd(qg, kg, vg, ag, bg, scale=scale, dev_err=err)
        oc = orth.xattn_fwd(qcg, pg, kg, vg, acg, bcg, scale=scale, dev_err=err)
        lse = lsec = None
    got = orth.attn_bwd(qg, kg, vg, ag, bg, o, bf(dO), qcg, pg, acg, bcg, oc, bf(dOc), scale=scale, lse=lse,
                        lsec=lsec, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = [t.cpu().numpy().astype(np.float64) for t in got]
    ref = _reference((q, k, v, a, b, dO, qc, pos, dOc, ac, bc, scale), 128)
    for name, gg, r in zip(LAYER_NAMES, got, ref):
        _assert_grad(gg, r, f"{name} with keys beyond fp16")
