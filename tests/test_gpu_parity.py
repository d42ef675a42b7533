"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs, at sizes the oracle finishes in seconds that still span
several tiles and a ragged tail, plus the edge cases of the operator.  Bar:
max-abs 1e-2 and mean-abs 1e-3 on bf16 outputs; bit-exact for the KV cache and
for mask / position handling."""
import math

import numpy as np
import pytest
import torch

import long_context_attention_orthros_gb300 as orth
import oracle
from synthetic import (CONFIGS, SEEDS, PrefillConfig, bf16_bits, make_prefill, normal_bf16,
                       reduced, scale_offset)
from tests.gpu_util import assert_parity, bf, bits, dev, f32, i32, val

pytestmark = pytest.mark.gpu


def _run_prefill(inp, window=None):
    cfg = inp.cfg
    w = cfg.window if window is None else window
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    q_all = bf(inp.q_raw)
    k, v = bf(inp.k), bf(inp.v)
    o = orth.swa_fwd(q_all, k, v, f32(inp.alpha), f32(inp.beta), window=w, scale=cfg.scale,
                     dev_err=err)
    qc = q_all[:, cfg.T:] if cfg.appended else bf(inp.qc_raw)
    oc = orth.xattn_fwd(qc, i32(inp.pos), k, v, f32(inp.alpha_c), f32(inp.beta_c),
                        scale=cfg.scale, dev_err=err)
    torch.cuda.synchronize()
    return o, oc, int(err.item())


def _check_prefill(inp, window=None):
    cfg = inp.cfg
    w = cfg.window if window is None else window
    o, oc, err = _run_prefill(inp, window)
    assert err == 0
    ref_o = oracle.swa(np.ascontiguousarray(inp.q_base), inp.k, inp.v, inp.alpha, inp.beta, w,
                       cfg.scale)
    ref_oc = oracle.xattn(np.ascontiguousarray(inp.qc_raw), inp.pos, inp.k, inp.v, inp.alpha_c,
                          inp.beta_c, cfg.scale)
    assert_parity(val(o), ref_o, "base O")
    assert_parity(val(oc), ref_oc, "copy O'")


def test_tiny_prefill_config():
    """The tiny prefill workload at its full size (T=512, 2 q heads / 1 KV head, d=64)."""
    cfg = CONFIGS["tiny_prefill"]
    _check_prefill(make_prefill(cfg, SEEDS[cfg.name]))


@pytest.mark.parametrize("B,T,Hq,Hkv,d,w", [
    (2, 1000, 32, 8, 128, 128),   # 8B-class heads, ragged tail (1000 = 31*32 + 8)
    (1, 777, 8, 4, 64, 128),      # G=2, d=64
    (1, 300, 4, 4, 128, 128),     # G=1
    (1, 257, 16, 2, 128, 128),    # G=8
    (1, 200, 16, 1, 64, 128),     # G=16
    (2, 333, 8, 2, 128, 1),       # w=1
    (1, 500, 8, 2, 128, 7),       # narrow window
    (1, 640, 8, 2, 128, 200),     # wider band, still resident
    (1, 600, 8, 2, 128, 600),     # w >= T: full causal, streamed K/V blocks
    (1, 5, 4, 1, 128, 128),       # T smaller than a tile
])
def test_prefill_parity(B, T, Hq, Hkv, d, w):
    cfg = PrefillConfig("case", B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, window=w)
    _check_prefill(make_prefill(cfg, 1000 + T), window=w)


def test_sft_appended_shuffled_copies():
    """SFT layout at reduced size: copies of the last positions appended after the base
    tokens in one buffer, original positions in shuffled order (many-row path)."""
    cfg = reduced(CONFIGS["sft_16k"], B=2, T=1500, T_out=200)
    _check_prefill(make_prefill(cfg, 77))


def test_copies_mixed_positions_and_duplicates():
    cfg = PrefillConfig("mixed", B=2, T=900, Hq=8, Hkv=2, d=128, T_out=7)
    inp = make_prefill(cfg, 5)
    inp.pos[:] = np.array([[0, 1, 63, 64, 899, 899, 450], [898, 5, 5, 127, 128, 300, 0]], np.int32)
    _check_prefill(inp)


def test_needle_keys_sharp_peaks():
    """Scaled key rows at seeded positions (the 1M workload's recipe) at reduced size."""
    cfg = reduced(CONFIGS["prefill_1m"], T=4096, needle_frac=0.002)
    _check_prefill(make_prefill(cfg, 9))


def test_bad_position_sets_error_and_zero_row():
    cfg = PrefillConfig("bad", B=1, T=300, Hq=4, Hkv=1, d=128, T_out=3)
    inp = make_prefill(cfg, 3)
    inp.pos[0] = [10, 300, 299]
    _o, oc, err = _run_prefill(inp)
    assert err & orth.DEVERR_POSITION
    got = val(oc)
    assert (got[0, 1] == 0).all()
    ok = [0, 2]
    ref = oracle.xattn(np.ascontiguousarray(inp.qc_raw[:, ok]), inp.pos[:, ok], inp.k, inp.v,
                       inp.alpha_c, inp.beta_c, cfg.scale)
    assert_parity(got[:, ok], ref, "valid copies next to a bad one")


def test_window_one_is_bit_exact():
    """w=1: every weight is exactly 1, so o_t equals v_t bit for bit."""
    cfg = PrefillConfig("w1", B=1, T=130, Hq=8, Hkv=2, d=128, window=1)
    inp = make_prefill(cfg, 4)
    o, _oc, _ = _run_prefill(inp, window=1)
    np.testing.assert_array_equal(bits(o), np.repeat(inp.v, cfg.Hq // cfg.Hkv, axis=2))


def test_mask_membership_is_exact():
    """K == 0 gives equal weights; a single non-zero value row j* makes o_t[0] exactly
    zero for rows whose window misses j* and non-zero for rows that contain it."""
    B, T, Hq, Hkv, d, w = 1, 700, 8, 2, 128, 128
    q = normal_bf16(1, "q_raw", (B, T, Hq, d))
    k = np.zeros((B, T, Hkv, d), np.uint16)
    for jstar in (0, 131, 500, 699):
        vf = np.zeros((B, T, Hkv, d), np.float32)
        vf[0, jstar, :, 0] = 1.0
        v = bf16_bits(vf)
        a, b = scale_offset(1, Hq, d)
        o = val(orth.swa_fwd(bf(q), bf(k), bf(v), f32(a), f32(b), window=w))
        t = np.arange(T)
        inside = (jstar <= t) & (jstar > t - w)
        seen = o[0, :, :, 0] != 0
        np.testing.assert_array_equal(seen, np.repeat(inside[:, None], Hq, axis=1))
        # copies: a copy at position p sees j* iff j* <= p
        pos = np.array([[jstar - 1 if jstar else 0, jstar, T - 1]], np.int32)
        qc = normal_bf16(2, "qc_raw", (B, 3, Hq, d))
        oc = val(orth.xattn_fwd(bf(qc), i32(pos), bf(k), bf(v), f32(a), f32(b)))
        seen_c = oc[0, :, :, 0] != 0
        np.testing.assert_array_equal(seen_c, np.repeat((jstar <= pos[0])[:, None], Hq, axis=1))


def test_copy_permutation_is_bit_exact():
    """Permuting the physical order of the copies (with their positions) permutes the
    outputs bit for bit (masks follow original positions)."""
    cfg = PrefillConfig("perm", B=2, T=1200, Hq=32, Hkv=8, d=128, T_out=40, positions="shuffled")
    inp = make_prefill(cfg, 8)
    k, v = bf(inp.k), bf(inp.v)
    oc1 = orth.xattn_fwd(bf(inp.qc_raw), i32(inp.pos), k, v, f32(inp.alpha_c), f32(inp.beta_c))
    perm = np.random.default_rng(3).permutation(cfg.T_out)
    oc2 = orth.xattn_fwd(bf(np.ascontiguousarray(inp.qc_raw[:, perm])),
                         i32(np.ascontiguousarray(inp.pos[:, perm])), k, v,
                         f32(inp.alpha_c), f32(inp.beta_c))
    np.testing.assert_array_equal(bits(oc2), bits(oc1)[:, perm])


def test_copy_equals_base_causal_row_when_streams_coincide():
    """alpha'=alpha, beta'=beta, x'=x: the copy at t equals the w >= T base stream at t."""
    B, T, Hq, Hkv, d = 1, 400, 8, 2, 128
    q = normal_bf16(6, "q_raw", (B, T, Hq, d))
    k = normal_bf16(6, "k", (B, T, Hkv, d))
    v = normal_bf16(6, "v", (B, T, Hkv, d))
    a, b = scale_offset(6, Hq, d)
    full = val(orth.swa_fwd(bf(q), bf(k), bf(v), f32(a), f32(b), window=T))
    pos = np.array([[0, 57, 128, 399]], np.int32)
    oc = val(orth.xattn_fwd(bf(np.ascontiguousarray(q[:, pos[0]])), i32(pos), bf(k), bf(v),
                            f32(a), f32(b)))
    assert np.abs(oc[0] - full[0, pos[0]]).max() <= 2e-2


def test_output_alignment_paths_agree():
    """Output rows go out as whole 32-byte sectors when the output is 32-byte aligned and
    as 16-byte pieces otherwise; both paths hold the same bits and meet the oracle."""
    cfg = PrefillConfig("case", B=2, T=700, Hq=32, Hkv=8, d=128, window=128)
    inp = make_prefill(cfg, 4242)
    q, k, v = bf(inp.q_raw), bf(inp.k), bf(inp.v)
    a, b = f32(inp.alpha), f32(inp.beta)
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    o_aligned = orth.swa_fwd(q, k, v, a, b, window=cfg.window, scale=cfg.scale, dev_err=err)
    n = cfg.B * cfg.T * cfg.Hq * cfg.d
    buf = torch.zeros(n + 8, dtype=torch.bfloat16, device=dev())
    o_off = buf[8:].view(cfg.B, cfg.T, cfg.Hq, cfg.d)  # 16 bytes past a 32-byte boundary
    orth.swa_fwd(q, k, v, a, b, window=cfg.window, scale=cfg.scale, out=o_off, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert o_off.data_ptr() % 32 == 16
    assert torch.equal(o_off.view(torch.int16), o_aligned.view(torch.int16))
    ref = oracle.swa(np.ascontiguousarray(inp.q_base), inp.k, inp.v, inp.alpha, inp.beta, cfg.window,
                     cfg.scale)
    assert_parity(val(o_off), ref, "base O, 16-byte stores")
