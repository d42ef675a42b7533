"""Pins for the fp64 oracle, checked against things other than the oracle itself:
library routines (PyTorch CPU scaled-dot-product attention in float64), closed
forms, the pages' teaching example, brute force on tiny inputs, and invariants
the pages fix (Orthros, Sec. 2.3-2.5 of the close-reading notes: Eqs. (4)-(5),
dependency isolation, original-position masks, the four modes).

Each pin is chosen so that a plausible slip in the oracle (window off by one,
a dropped beta, alpha applied to the key, the wrong GQA head, values and keys
swapped, a missing max-subtraction or normalisation, the copy masked by its
physical slot, attend-before-append in decode) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from synthetic import bf16_bits, bf16_to_f32, normal_bf16, scale_offset

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_inputs(seed, B, T, Hq, Hkv, d):
    q = normal_bf16(seed, "q_raw", (B, T, Hq, d))
    k = normal_bf16(seed, "k", (B, T, Hkv, d))
    v = normal_bf16(seed, "v", (B, T, Hkv, d))
    a, b = scale_offset(seed, Hq, d)
    return q, k, v, a, b


def _sdpa(q64, k64, v64, mask, scale):
    """Library reference: torch SDPA in float64 on the CPU.  q64 [B,T,Hq,d];
    k64/v64 [B,S,Hkv,d]; GQA by repeat_interleave (head h -> kv head h // group)."""
    Hq, Hkv = q64.shape[2], k64.shape[2]
    kq = torch.from_numpy(k64).repeat_interleave(Hq // Hkv, dim=2)
    vq = torch.from_numpy(v64).repeat_interleave(Hq // Hkv, dim=2)
    out = F.scaled_dot_product_attention(
        torch.from_numpy(q64).transpose(1, 2), kq.transpose(1, 2), vq.transpose(1, 2),
        attn_mask=None if mask is None else torch.from_numpy(mask), scale=scale)
    return out.transpose(1, 2).numpy()


def _w(x):
    return bf16_to_f32(x).astype(np.float64)


def _band(T, w):
    t = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    return (j <= t) & (j > t - w)


@pytest.mark.parametrize("B,T,Hq,Hkv,d,w", [
    (1, 1, 1, 1, 8, 1), (1, 37, 2, 1, 16, 5), (2, 130, 4, 2, 32, 128),
    (1, 300, 8, 2, 64, 128), (2, 200, 4, 4, 16, 64), (1, 257, 6, 3, 8, 300)])
def test_swa_equals_sdpa_with_band_mask(B, T, Hq, Hkv, d, w):
    """Eq. (4) with scale-offset == library SDPA over the band mask W_t (GQA expanded)."""
    q, k, v, a, b = _rand_inputs(100 + T, B, T, Hq, Hkv, d)
    s = 1 / math.sqrt(d)
    o = oracle.swa(q, k, v, a, b, w, s)
    q64 = _w(q) * a.astype(np.float64) + b.astype(np.float64)
    ref = _sdpa(q64, _w(k), _w(v), _band(T, w), s)
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


def test_swa_rows_equal_sdpa_at_the_sampled_rows():
    """The sampled-row form (the reference of the full-size GPU tests) == library SDPA over the
    band mask at those rows: both batch entries, the first and last rows, rows at the window
    edge, a repeated row, in arbitrary order."""
    B, T, Hq, Hkv, d, w = 2, 70, 4, 2, 16, 9
    q, k, v, a, b = _rand_inputs(111, B, T, Hq, Hkv, d)
    s = 1 / math.sqrt(d)
    bi = np.array([0, 1, 1, 0, 1, 0, 1], np.int64)
    ti = np.array([0, T - 1, 8, 9, 9, T - 1, 0], np.int64)
    got = oracle.swa_rows(q, k, v, a, b, w, s, bi, ti)
    q64 = _w(q) * a.astype(np.float64) + b.astype(np.float64)
    ref = _sdpa(q64, _w(k), _w(v), _band(T, w), s)
    np.testing.assert_allclose(got, ref[bi, ti], rtol=0, atol=1e-12)


def test_swa_window_ge_T_is_full_causal():
    """With w >= T the sliding window covers all of 1..t: plain causal attention."""
    B, T, Hq, Hkv, d = 2, 96, 4, 1, 32
    q, k, v, a, b = _rand_inputs(7, B, T, Hq, Hkv, d)
    s = 1 / math.sqrt(d)
    o = oracle.swa(q, k, v, np.ones_like(a), np.zeros_like(b), 128, s)
    kq = torch.from_numpy(_w(k)).repeat_interleave(Hq, dim=2)
    vq = torch.from_numpy(_w(v)).repeat_interleave(Hq, dim=2)
    ref = F.scaled_dot_product_attention(torch.from_numpy(_w(q)).transpose(1, 2),
                                         kq.transpose(1, 2), vq.transpose(1, 2),
                                         is_causal=True).transpose(1, 2).numpy()
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


def test_rows_before_window_fills_equal_causal_rows():
    """Rows t < w see all of 0..t, so they equal the full-causal rows; later rows differ."""
    B, T, Hq, Hkv, d, w = 1, 80, 2, 1, 16, 32
    q, k, v, a, b = _rand_inputs(8, B, T, Hq, Hkv, d)
    s = 1 / math.sqrt(d)
    o_w = oracle.swa(q, k, v, a, b, w, s)
    o_full = oracle.swa(q, k, v, a, b, T, s)
    np.testing.assert_array_equal(o_w[:, :w], o_full[:, :w])
    assert np.abs(o_w[:, w:] - o_full[:, w:]).max() > 1e-3


@pytest.mark.parametrize("T,w,d", [(300, 128, 64), (50, 7, 8), (5, 128, 4)])
def test_zero_keys_reveal_the_exact_window(T, w, d):
    """K == 0 makes every weight equal: o_t is the mean of v over W_t.  With
    v_j = (j mod 128, j div 128, 1, 0, ...) (exact in bf16), 128*o[1] + o[0] is the
    mean of the window's indices, (lo + t) / 2 with lo = max(0, t-w+1), and o[2]
    is exactly 1."""
    B, Hq, Hkv = 1, 2, 1
    q = normal_bf16(3, "q_raw", (B, T, Hq, d))
    k = np.zeros((B, T, Hkv, d), np.uint16)
    vf = np.zeros((B, T, Hkv, d), np.float32)
    vf[0, :, 0, 0] = np.arange(T) % 128
    vf[0, :, 0, 1] = np.arange(T) // 128
    vf[0, :, 0, 2] = 1
    v = bf16_bits(vf)
    assert np.array_equal(bf16_to_f32(v), vf)
    a, b = scale_offset(3, Hq, d)
    o = oracle.swa(q, k, v, a, b, w, 0.5)
    t = np.arange(T)
    lo = np.maximum(0, t - w + 1)
    for h in range(Hq):
        np.testing.assert_allclose(128 * o[0, :, h, 1] + o[0, :, h, 0], (lo + t) / 2,
                                   rtol=0, atol=1e-11)
        np.testing.assert_allclose(o[0, :, h, 2], 1.0, rtol=0, atol=1e-14)
        np.testing.assert_array_equal(o[0, :, h, 3:], 0.0)


def test_window_one_is_identity_on_values():
    """w = 1: each position attends only to itself, o_t = v_t exactly."""
    B, T, Hq, Hkv, d = 2, 40, 4, 2, 16
    q, k, v, a, b = _rand_inputs(9, B, T, Hq, Hkv, d)
    o = oracle.swa(q, k, v, a, b, 1, 0.25)
    vq = np.repeat(_w(v), Hq // Hkv, axis=2)
    np.testing.assert_array_equal(o, vq)


def test_constant_values_give_that_constant():
    """Weights sum to one: if every v_j = c then o_t = c, for any keys and queries."""
    B, T, Hq, Hkv, d = 1, 70, 2, 1, 8
    q, k, _, a, b = _rand_inputs(10, B, T, Hq, Hkv, d)
    c = np.linspace(-2, 2, d).astype(np.float32)
    v = bf16_bits(np.broadcast_to(c, (B, T, Hkv, d)))
    o = oracle.swa(q, k, v, a, b, 16, 0.3)
    np.testing.assert_allclose(o, np.broadcast_to(_w(v)[0, 0, 0], o.shape), rtol=0, atol=1e-14)


def test_scale_offset_alpha_zero_leaves_only_beta():
    """alpha = 0: q = beta for every row, whatever Q_raw holds.  Pins that beta is
    added to the query (not the key) and that alpha multiplies Q_raw."""
    B, T, Hq, Hkv, d = 1, 60, 2, 1, 16
    q, k, v, _, b = _rand_inputs(11, B, T, Hq, Hkv, d)
    s = 0.25
    o1 = oracle.swa(q, k, v, np.zeros((Hq, d), np.float32), b, 8, s)
    q2 = normal_bf16(12, "q_raw", (B, T, Hq, d))
    o2 = oracle.swa(q2, k, v, np.zeros((Hq, d), np.float32), b, 8, s)
    np.testing.assert_array_equal(o1, o2)
    qb = np.broadcast_to(b.astype(np.float64), (B, T, Hq, d)).copy()
    ref = _sdpa(qb, _w(k), _w(v), _band(T, 8), s)
    np.testing.assert_allclose(o1, ref, rtol=0, atol=1e-12)


def test_scale_offset_is_per_head():
    """alpha/beta are [Hq, d]: head h uses row h (checked with rows that differ)."""
    B, T, Hq, Hkv, d = 1, 33, 4, 2, 8
    q, k, v, a, b = _rand_inputs(13, B, T, Hq, Hkv, d)
    s = 1 / math.sqrt(d)
    o = oracle.swa(q, k, v, a, b, 10, s)
    for h in range(Hq):
        q64 = _w(q[:, :, h:h + 1]) * a[h].astype(np.float64) + b[h].astype(np.float64)
        ref = _sdpa(q64, _w(k[:, :, h // 2:h // 2 + 1]), _w(v[:, :, h // 2:h // 2 + 1]),
                    _band(T, 10), s)
        np.testing.assert_allclose(o[:, :, h:h + 1], ref, rtol=0, atol=1e-12)


def test_brute_force_triple_loop_tiny():
    """Brute force in pure Python on a tiny case (explicit sums, no vector ops)."""
    B, T, Hq, Hkv, d, w = 1, 9, 2, 1, 3, 4
    q, k, v, a, b = _rand_inputs(14, B, T, Hq, Hkv, d)
    s = 0.7
    o = oracle.swa(q, k, v, a, b, w, s)
    qf, kf, vf = _w(q), _w(k), _w(v)
    for t in range(T):
        for h in range(Hq):
            qq = [qf[0, t, h, e] * float(a[h, e]) + float(b[h, e]) for e in range(d)]
            js = list(range(max(0, t - w + 1), t + 1))
            lg = [s * sum(qq[e] * kf[0, j, 0, e] for e in range(d)) for j in js]
            m = max(lg)
            ws = [math.exp(x - m) for x in lg]
            z = sum(ws)
            for e in range(d):
                ref = sum(ws[i] * vf[0, j, 0, e] for i, j in enumerate(js)) / z
                assert abs(o[0, t, h, e] - ref) < 1e-13


def test_large_logits_do_not_overflow():
    """Softmax is shift-invariant; logits near 700 must not overflow (max subtraction)."""
    B, T, Hq, Hkv, d = 1, 20, 1, 1, 4
    qf = np.zeros((B, T, Hq, d), np.float32)
    qf[..., 0] = 32.0
    kf = np.zeros((B, T, Hkv, d), np.float32)
    kf[0, :, 0, 0] = 32.0 + np.arange(T) % 3
    v = normal_bf16(15, "v", (B, T, Hkv, d))
    o = oracle.swa(bf16_bits(qf), bf16_bits(kf), v, np.ones((Hq, d), np.float32),
                   np.zeros((Hq, d), np.float32), 8, 0.7)
    assert np.isfinite(o).all()
    ref = _sdpa(_w(bf16_bits(qf)), _w(bf16_bits(kf)), _w(v), _band(T, 8), 0.7)
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-10)


# ----------------------------------------------------------------- copies (Eq. 5)

def test_copy_equals_causal_row_when_streams_coincide():
    """With alpha'=alpha, beta'=beta and x'=x, the copy at t equals row t of
    standard causal attention (Eq. 5 reads all j <= t)."""
    B, T, Hq, Hkv, d = 2, 150, 4, 2, 32
    q, k, v, a, b = _rand_inputs(20, B, T, Hq, Hkv, d)
    s = 1 / math.sqrt(d)
    pos = np.array([[149, 0, 77, 128], [5, 149, 149, 60]], np.int32)
    qc = np.stack([q[bb, pos[bb]] for bb in range(B)])
    oc = oracle.xattn(qc, pos, k, v, a, b, s)
    q64 = _w(q) * a.astype(np.float64) + b.astype(np.float64)
    full = _sdpa(q64, _w(k), _w(v), _band(T, T + 1), s)
    for bb in range(B):
        np.testing.assert_allclose(oc[bb], full[bb, pos[bb]], rtol=0, atol=1e-12)
    # and it is the w >= T base stream at that row
    o_full = oracle.swa(q, k, v, a, b, T, s)
    for bb in range(B):
        np.testing.assert_allclose(oc[bb], o_full[bb, pos[bb]], rtol=0, atol=1e-13)


def test_copy_mask_uses_original_position_not_slot():
    """Algorithm 2 appends copies at the tensor tail; the mask must follow the
    original position.  Permuting the physical order (with pos) permutes the
    outputs and changes nothing else, bit for bit."""
    B, T, Hq, Hkv, d, n = 2, 120, 4, 1, 16, 11
    _, k, v, _, _ = _rand_inputs(21, B, T, Hq, Hkv, d)
    qc = normal_bf16(21, "qc_raw", (B, n, Hq, d))
    ac, bc = scale_offset(21, Hq, d, prefix="_c")
    g = np.random.default_rng(5)
    pos = np.stack([g.choice(T, n, replace=False) for _ in range(B)]).astype(np.int32)
    oc = oracle.xattn(qc, pos, k, v, ac, bc, 0.25)
    perm = g.permutation(n)
    oc_p = oracle.xattn(qc[:, perm], pos[:, perm], k, v, ac, bc, 0.25)
    np.testing.assert_array_equal(oc_p, oc[:, perm])
    # a copy whose query is placed in slot 0 but whose position is 50 reads keys 0..50
    kz = np.zeros_like(k)
    vf = np.zeros((B, T, Hkv, d), np.float32)
    vf[:, :, 0, 0] = np.arange(T)
    one = oracle.xattn(qc[:, :1], np.array([[50], [3]], np.int32), kz, bf16_bits(vf), ac, bc, 0.25)
    np.testing.assert_allclose(one[0, 0, :, 0], 25.0, atol=1e-12)
    np.testing.assert_allclose(one[1, 0, :, 0], 1.5, atol=1e-12)


def test_copies_allow_duplicates_and_position_zero():
    B, T, Hq, Hkv, d = 1, 64, 2, 1, 8
    _, k, v, _, _ = _rand_inputs(22, B, T, Hq, Hkv, d)
    qc = normal_bf16(22, "qc_raw", (B, 3, Hq, d))
    qc[:, 1] = qc[:, 0]
    ac, bc = scale_offset(22, Hq, d, prefix="_c")
    oc = oracle.xattn(qc, np.array([[9, 9, 0]], np.int32), k, v, ac, bc, 0.3)
    np.testing.assert_array_equal(oc[:, 0], oc[:, 1])
    np.testing.assert_array_equal(oc[0, 2], np.repeat(_w(v)[0, 0], Hq, axis=0))


def test_copy_rejects_out_of_range_positions():
    B, T, Hq, Hkv, d = 1, 16, 2, 1, 8
    _, k, v, _, _ = _rand_inputs(23, B, T, Hq, Hkv, d)
    qc = normal_bf16(23, "qc_raw", (B, 1, Hq, d))
    ac, bc = scale_offset(23, Hq, d, prefix="_c")
    for bad in (-1, T):
        with pytest.raises(ValueError):
            oracle.xattn(qc, np.array([[bad]], np.int32), k, v, ac, bc, 0.3)


# ----------------------------------------------------------------- decode (Sec. 3.2)

def _decode_run(T0, steps, B=2, Hq=4, Hkv=2, d=16, w=8, seed=30):
    L = T0 + steps
    T = L
    q, k, v, a, b = _rand_inputs(seed, B, T, Hq, Hkv, d)
    qc = normal_bf16(seed, "qc_raw", (B, T, Hq, d))
    ac, bc = scale_offset(seed, Hq, d, prefix="_c")
    kc = np.full((B, L, Hkv, d), 0x7FC0, np.uint16)
    vc = np.full((B, L, Hkv, d), 0x7FC0, np.uint16)
    kc[:, :T0], vc[:, :T0] = k[:, :T0], v[:, :T0]
    cl = np.full((B,), T0, np.int32)
    outs = []
    for i in range(steps):
        p = T0 + i
        o, oc = oracle.decode_step(q[:, p], qc[:, p], k[:, p], v[:, p], kc, vc, cl,
                                   a, b, ac, bc, w, 1 / math.sqrt(d))
        outs.append((o, oc))
    return (q, k, v, a, b, qc, ac, bc), kc, vc, cl, outs


def test_decode_equals_prefill_at_appended_positions():
    """Decoding token by token gives the prefill result at each appended position,
    for the base output (Eq. 4) and for the copy (Eq. 5) (the [A,B,C] -> D, D' example)."""
    T0, steps, w, d = 20, 12, 8, 16
    (q, k, v, a, b, qc, ac, bc), kc, vc, cl, outs = _decode_run(T0, steps, w=w, d=d)
    s = 1 / math.sqrt(d)
    o_pre = oracle.swa(q, k, v, a, b, w, s)
    B = q.shape[0]
    pos = np.tile(np.arange(T0, T0 + steps, dtype=np.int32), (B, 1))
    oc_pre = oracle.xattn(np.stack([qc[bb, pos[bb]] for bb in range(B)]), pos, k, v, ac, bc, s)
    for i, (o, oc) in enumerate(outs):
        np.testing.assert_allclose(o, o_pre[:, T0 + i], rtol=0, atol=1e-13)
        np.testing.assert_allclose(oc, oc_pre[:, i], rtol=0, atol=1e-13)
    # cache after n steps = initial cache + appended rows, bit for bit
    np.testing.assert_array_equal(kc, k)
    np.testing.assert_array_equal(vc, v)
    np.testing.assert_array_equal(cl, T0 + steps)


def test_decode_copy_never_writes_cache_and_is_isolated():
    """Perturbing the copy's query or alpha'/beta' leaves o, the cache and cache_len
    bit-identical (output copies never write K/V, Sec. 2.4)."""
    B, Hq, Hkv, d, L, T0 = 1, 4, 1, 16, 40, 30
    k = normal_bf16(31, "k", (B, L, Hkv, d))
    v = normal_bf16(31, "v", (B, L, Hkv, d))
    a, b = scale_offset(31, Hq, d)
    ac, bc = scale_offset(31, Hq, d, prefix="_c")
    qn = normal_bf16(31, "q_new", (B, Hq, d))
    kn = normal_bf16(31, "k_new", (B, Hkv, d))
    vn = normal_bf16(31, "v_new", (B, Hkv, d))
    res = []
    for qc_seed, acs in ((1, 1.0), (2, 3.0)):
        kc, vc = k.copy(), v.copy()
        kc[:, T0:] = 0x7FC0
        vc[:, T0:] = 0x7FC0
        cl = np.full((B,), T0, np.int32)
        qcn = normal_bf16(qc_seed, "qc_new", (B, Hq, d))
        o, oc = oracle.decode_step(qn, qcn, kn, vn, kc, vc, cl, a, b, ac * acs, bc * acs, 16, 0.25)
        res.append((o, oc, kc, vc, cl))
    np.testing.assert_array_equal(res[0][0], res[1][0])
    for i in (2, 3, 4):
        np.testing.assert_array_equal(res[0][i], res[1][i])
    assert np.abs(res[0][1] - res[1][1]).max() > 1e-3


def test_decode_reads_only_rows_below_cache_len():
    """Unused cache rows hold bf16 NaN; a correct step never touches them."""
    (_, _, _, _, _, _, _, _), kc, vc, cl, outs = _decode_run(10, 3)
    for o, oc in outs:
        assert np.isfinite(o).all() and np.isfinite(oc).all()


# ----------------------------------------------------------------- the pages' example

def _frac(rows):
    return np.array([n / dd for n, dd in rows], np.float64)


def test_golden_abc_teaching_example():
    """Sec. 2.4: prompt [A,B,C]; C' reads K_A, K_B, K_C; then D, D' in decode."""
    g = json.load(open(os.path.join(GOLDEN, "abc_teaching_example.json")))
    d, w = g["d"], g["window"]
    T = 3
    vals = np.array(g["prompt_values"], np.float32).reshape(1, T, 1, d)
    k = np.zeros((1, T, 1, d), np.uint16)
    v = bf16_bits(vals)
    q = normal_bf16(40, "q_raw", (1, T, 1, d))
    a, b = scale_offset(40, 1, d)
    ac, bc = scale_offset(40, 1, d, prefix="_c")
    s = 1 / math.sqrt(d)
    o = oracle.swa(q, k, v, a, b, w, s)
    ex = g["expected"]
    for t, name in enumerate(("base_A", "base_B", "base_C")):
        np.testing.assert_allclose(o[0, t, 0], _frac(ex[name]), rtol=0, atol=1e-15)
    qc = normal_bf16(40, "qc_raw", (1, 1, 1, d))
    oc = oracle.xattn(qc, np.array([[2]], np.int32), k, v, ac, bc, s)
    np.testing.assert_allclose(oc[0, 0, 0], _frac(ex["copy_C"]), rtol=0, atol=1e-15)
    # decode D: append, then D reads its window {C, D}, D' reads {A, B, C, D}
    L = 4
    kc = np.zeros((1, L, 1, d), np.uint16)
    vc = np.full((1, L, 1, d), 0x7FC0, np.uint16)
    vc[:, :T] = v
    cl = np.array([T], np.int32)
    vD = bf16_bits(np.array(g["decode_value"], np.float32).reshape(1, 1, d))
    o_d, oc_d = oracle.decode_step(q[:, 0], qc[:, 0], np.zeros((1, 1, d), np.uint16), vD,
                                   kc, vc, cl, a, b, ac, bc, w, s)
    np.testing.assert_allclose(o_d[0, 0], _frac(ex["decode_base_D"]), rtol=0, atol=1e-15)
    np.testing.assert_allclose(oc_d[0, 0], _frac(ex["decode_copy_D"]), rtol=0, atol=1e-15)
    np.testing.assert_array_equal(vc[0, 3], vD[0])
    assert cl[0] == 4
    # weighted variant: logits 0, 1, 2 exactly
    kf = np.zeros((1, T, 1, d), np.float32)
    kf[0, :, 0, 0] = [0, 1, 2]
    qcw = bf16_bits(np.array([1, 0, 0, 0], np.float32).reshape(1, 1, 1, d))
    oc_w = oracle.xattn(qcw, np.array([[2]], np.int32), bf16_bits(kf), v,
                        np.array([[2, 1, 1, 1]], np.float32), np.zeros((1, d), np.float32), s)
    e = np.exp(np.array(g["weighted"]["copy_logits"], np.float64))
    np.testing.assert_allclose(oc_w[0, 0, 0, :3], e / e.sum(), rtol=0, atol=1e-15)


# ---------------------------------------------------------------- gradient of Eq. (4)

def _autograd_swa_grads(q, k, v, a, b, dO, w, scale):
    """Library reference: torch autograd through float64 SDPA with the band mask and the
    scale-offset q = x * alpha + beta, for the loss sum(dO * o)."""
    x = torch.from_numpy(_w(q)).requires_grad_(True)
    kk = torch.from_numpy(_w(k)).requires_grad_(True)
    vv = torch.from_numpy(_w(v)).requires_grad_(True)
    al = torch.from_numpy(a.astype(np.float64)).requires_grad_(True)
    be = torch.from_numpy(b.astype(np.float64)).requires_grad_(True)
    Hq, Hkv = q.shape[2], k.shape[2]
    qq = x * al + be
    kq = kk.repeat_interleave(Hq // Hkv, dim=2)
    vq = vv.repeat_interleave(Hq // Hkv, dim=2)
    mask = torch.from_numpy(_band(q.shape[1], w))
    o = F.scaled_dot_product_attention(qq.transpose(1, 2), kq.transpose(1, 2), vq.transpose(1, 2),
                                       attn_mask=mask, scale=scale).transpose(1, 2)
    (o * torch.from_numpy(_w(dO))).sum().backward()
    return [t.grad.numpy() for t in (x, kk, vv, al, be)]


@pytest.mark.parametrize("B,T,Hq,Hkv,d,w", [
    (1, 9, 1, 1, 8, 3), (1, 40, 4, 2, 16, 7), (2, 33, 4, 1, 8, 128), (1, 70, 8, 2, 32, 16),
])
def test_swa_gradient_equals_autograd(B, T, Hq, Hkv, d, w):
    q, k, v, a, b = _rand_inputs(60 + T, B, T, Hq, Hkv, d)
    dO = normal_bf16(60 + T, "dO", (B, T, Hq, d))
    scale = 1.0 / math.sqrt(d)
    got = oracle.swa_bwd(q, k, v, a, b, dO, w, scale)
    ref = _autograd_swa_grads(q, k, v, a, b, dO, w, scale)
    for name, g, r in zip(("dq_raw", "dk", "dv", "dalpha", "dbeta"), got, ref):
        np.testing.assert_allclose(g, r, rtol=1e-9, atol=1e-11, err_msg=name)


def test_swa_gradient_in_values_is_exact_finite_difference():
    """o is linear in V, so a one-ulp bf16 step of one value element changes
    L = sum(dO * o) by exactly dv times the step."""
    B, T, Hq, Hkv, d, w = 1, 12, 2, 1, 8, 5
    q, k, v, a, b = _rand_inputs(71, B, T, Hq, Hkv, d)
    dO = normal_bf16(71, "dO", (B, T, Hq, d))
    scale = 1.0 / math.sqrt(d)
    dv = oracle.swa_bwd(q, k, v, a, b, dO, w, scale)[2]
    L0 = (oracle.swa(q, k, v, a, b, w, scale) * _w(dO)).sum()
    for (t, e) in [(0, 0), (5, 3), (11, 7)]:
        v2 = v.copy()
        v2[0, t, 0, e] = np.uint16(int(v2[0, t, 0, e]) + 1)  # next bf16 value
        step = _w(v2)[0, t, 0, e] - _w(v)[0, t, 0, e]
        L1 = (oracle.swa(q, k, v2, a, b, w, scale) * _w(dO)).sum()
        assert abs((L1 - L0) / step - dv[0, t, 0, e]) <= 1e-9 * max(1.0, abs(dv[0, t, 0, e]))


def test_swa_gradient_window_one():
    """w = 1: o_t = v_t, so dv_t = the sum of dO_t over the query heads of the KV head
    and there is no gradient in q, k, alpha or beta."""
    q, k, v, a, b = _rand_inputs(72, 2, 10, 4, 2, 8)
    dO = normal_bf16(72, "dO", (2, 10, 4, 8))
    dq, dk, dv, da, db = oracle.swa_bwd(q, k, v, a, b, dO, 1, 0.3)
    g = _w(dO).reshape(2, 10, 2, 2, 8).sum(axis=3)
    np.testing.assert_array_equal(dv, g)
    for z in (dq, dk, da, db):
        assert not z.any()


# ---------------------------------------------------------------- gradient of Eq. (5)

def _autograd_xattn_grads(qc, pos, k, v, a, b, dOc, scale):
    """Library reference: torch autograd through float64 SDPA where copy i sees keys
    0..pos[b, i], with the copies' scale-offset, for the loss sum(dOc * oc)."""
    B, T_out, Hq, d = qc.shape
    T_kv, Hkv = k.shape[1], k.shape[2]
    x = torch.from_numpy(_w(qc)).requires_grad_(True)
    kk = torch.from_numpy(_w(k)).requires_grad_(True)
    vv = torch.from_numpy(_w(v)).requires_grad_(True)
    al = torch.from_numpy(a.astype(np.float64)).requires_grad_(True)
    be = torch.from_numpy(b.astype(np.float64)).requires_grad_(True)
    qq = x * al + be
    kq = kk.repeat_interleave(Hq // Hkv, dim=2)
    vq = vv.repeat_interleave(Hq // Hkv, dim=2)
    mask = torch.from_numpy(np.arange(T_kv)[None, None, :] <= pos[:, :, None])  # [B, T_out, T_kv]
    o = F.scaled_dot_product_attention(qq.transpose(1, 2), kq.transpose(1, 2), vq.transpose(1, 2),
                                       attn_mask=mask[:, None], scale=scale).transpose(1, 2)
    (o * torch.from_numpy(_w(dOc))).sum().backward()
    return [t.grad.numpy() for t in (x, kk, vv, al, be)]


@pytest.mark.parametrize("B,T_kv,T_out,Hq,Hkv,d", [
    (1, 9, 3, 1, 1, 8), (2, 40, 6, 4, 2, 16), (1, 70, 11, 8, 2, 32), (2, 25, 25, 4, 1, 8),
])
def test_xattn_gradient_equals_autograd(B, T_kv, T_out, Hq, Hkv, d):
    """Shuffled positions with duplicates, position 0 and the last position included."""
    _, k, v, _, _ = _rand_inputs(80 + T_kv, B, T_kv, Hq, Hkv, d)
    qc = normal_bf16(80 + T_kv, "qc_raw", (B, T_out, Hq, d))
    a, b = scale_offset(80 + T_kv, Hq, d, prefix="_c")
    g = np.random.default_rng(T_kv)
    pos = g.integers(0, T_kv, size=(B, T_out)).astype(np.int32)
    pos[:, 0] = 0
    pos[:, -1] = T_kv - 1
    if T_out > 2:
        pos[:, 1] = pos[:, 2]
    dOc = normal_bf16(80 + T_kv, "dOc", (B, T_out, Hq, d))
    scale = 1.0 / math.sqrt(d)
    got = oracle.xattn_bwd(qc, pos, k, v, a, b, dOc, scale)
    ref = _autograd_xattn_grads(qc, pos, k, v, a, b, dOc, scale)
    for name, gg, r in zip(("dqc_raw", "dk", "dv", "dalpha_c", "dbeta_c"), got, ref):
        np.testing.assert_allclose(gg, r, rtol=1e-9, atol=1e-11, err_msg=name)


def test_xattn_gradient_of_a_copy_at_every_position_is_the_causal_gradient():
    """Copies of every row in order, with the base query, scale-offset and output gradient,
    see exactly what base rows see when w >= T (Eq. (5) at pos = t is Eq. (4) with the
    window open), so the two gradients coincide."""
    B, T, Hq, Hkv, d = 2, 30, 4, 2, 16
    q, k, v, a, b = _rand_inputs(90, B, T, Hq, Hkv, d)
    dO = normal_bf16(90, "dO", (B, T, Hq, d))
    pos = np.tile(np.arange(T, dtype=np.int32), (B, 1))
    scale = 0.2
    base = oracle.swa_bwd(q, k, v, a, b, dO, T, scale)
    copy = oracle.xattn_bwd(q, pos, k, v, a, b, dO, scale)
    for name, x, y in zip(("dq_raw", "dk", "dv", "dalpha", "dbeta"), copy, base):
        np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-13, err_msg=name)


def test_xattn_gradient_in_values_is_exact_finite_difference():
    B, T_kv, T_out, Hq, Hkv, d = 1, 14, 4, 2, 1, 8
    _, k, v, _, _ = _rand_inputs(91, B, T_kv, Hq, Hkv, d)
    qc = normal_bf16(91, "qc_raw", (B, T_out, Hq, d))
    a, b = scale_offset(91, Hq, d, prefix="_c")
    pos = np.array([[13, 2, 7, 7]], np.int32)
    dOc = normal_bf16(91, "dOc", (B, T_out, Hq, d))
    scale = 1.0 / math.sqrt(d)
    dv = oracle.xattn_bwd(qc, pos, k, v, a, b, dOc, scale)[2]
    L0 = (oracle.xattn(qc, pos, k, v, a, b, scale) * _w(dOc)).sum()
    for (j, e) in [(0, 0), (2, 5), (7, 1), (13, 7)]:
        v2 = v.copy()
        v2[0, j, 0, e] = np.uint16(int(v2[0, j, 0, e]) + 1)
        step = _w(v2)[0, j, 0, e] - _w(v)[0, j, 0, e]
        L1 = (oracle.xattn(qc, pos, k, v2, a, b, scale) * _w(dOc)).sum()
        assert abs((L1 - L0) / step - dv[0, j, 0, e]) <= 1e-9 * max(1.0, abs(dv[0, j, 0, e]))


def test_xattn_gradient_position_zero():
    """A copy at position 0 sees only key 0: its output is v_0, so dv_0 gathers its dOc
    and nothing flows to q', k, alpha' or beta'."""
    _, k, v, _, _ = _rand_inputs(92, 1, 6, 4, 2, 8)
    qc = normal_bf16(92, "qc_raw", (1, 3, 4, 8))
    a, b = scale_offset(92, 4, 8, prefix="_c")
    dOc = normal_bf16(92, "dOc", (1, 3, 4, 8))
    pos = np.zeros((1, 3), np.int32)
    dq, dk, dv, da, db = oracle.xattn_bwd(qc, pos, k, v, a, b, dOc, 0.3)
    np.testing.assert_array_equal(dv[0, 0], _w(dOc)[0].reshape(3, 2, 2, 8).sum(axis=(0, 2)))
    assert not dv[0, 1:].any()
    for z in (dq, dk, da, db):
        assert not z.any()


# ---------------------------------------------------------------- row log-sum-exp of Eq. (4)

def test_swa_lse_of_zero_keys_is_log_of_window_size():
    """K = 0: every logit is 0, so lse_t = ln(min(t + 1, w)) exactly."""
    q, k, _, a, b = _rand_inputs(93, 2, 40, 4, 2, 16)
    k = np.zeros_like(k)
    got = oracle.swa_lse(q, k, a, b, 7, 0.25)
    n = np.minimum(np.arange(40) + 1, 7).astype(np.float64)
    np.testing.assert_allclose(got, np.broadcast_to(np.log(n)[None, :, None], got.shape), rtol=0, atol=1e-15)


@pytest.mark.parametrize("T,Hq,Hkv,d,w", [(30, 4, 2, 16, 5), (65, 8, 2, 32, 128), (50, 2, 2, 8, 1)])
def test_swa_lse_equals_scipy_logsumexp(T, Hq, Hkv, d, w):
    """Library reference: scipy's logsumexp over the band of float64 logits from einsum."""
    from scipy.special import logsumexp
    q, k, _, a, b = _rand_inputs(94 + T, 1, T, Hq, Hkv, d)
    scale = 1.0 / math.sqrt(d)
    qq = _w(q) * a.astype(np.float64) + b.astype(np.float64)
    kq = np.repeat(_w(k), Hq // Hkv, axis=2)
    logits = np.einsum("bthd,bshd->bhts", qq, kq) * scale
    band = _band(T, w)  # True where key s is in row t's window
    ref = logsumexp(np.where(band[None, None], logits, -np.inf), axis=-1).transpose(0, 2, 1)
    np.testing.assert_allclose(oracle.swa_lse(q, k, a, b, w, scale), ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- row log-sum-exp of Eq. (5)

def test_xattn_lse_of_zero_keys_is_log_of_position_count():
    """K = 0: every logit is 0, so a copy at position p has lse = ln(p + 1) exactly."""
    _, k, _, _, _ = _rand_inputs(95, 2, 50, 4, 2, 16)
    k = np.zeros_like(k)
    qc = normal_bf16(95, "qc_raw", (2, 6, 4, 16))
    a, b = scale_offset(95, 4, 16, prefix="_c")
    pos = np.array([[0, 49, 7, 7, 20, 1], [3, 0, 48, 12, 49, 5]], np.int32)
    got = oracle.xattn_lse(qc, pos, k, a, b, 0.3)
    want = np.broadcast_to(np.log(pos.astype(np.float64) + 1.0)[:, :, None], got.shape)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-15)


@pytest.mark.parametrize("T_kv,T_out,Hq,Hkv,d", [(40, 9, 4, 2, 16), (70, 5, 8, 1, 32)])
def test_xattn_lse_equals_scipy_logsumexp(T_kv, T_out, Hq, Hkv, d):
    """Library reference: scipy's logsumexp over keys 0..pos of float64 logits from einsum."""
    from scipy.special import logsumexp
    _, k, _, _, _ = _rand_inputs(96 + T_kv, 1, T_kv, Hq, Hkv, d)
    qc = normal_bf16(96 + T_kv, "qc_raw", (1, T_out, Hq, d))
    a, b = scale_offset(96 + T_kv, Hq, d, prefix="_c")
    pos = np.random.default_rng(T_kv).integers(0, T_kv, size=(1, T_out)).astype(np.int32)
    scale = 1.0 / math.sqrt(d)
    qq = _w(qc) * a.astype(np.float64) + b.astype(np.float64)
    kq = np.repeat(_w(k), Hq // Hkv, axis=2)
    logits = np.einsum("bihd,bshd->bhis", qq, kq) * scale
    seen = np.arange(T_kv)[None, None, :] <= pos[:, :, None]  # [1, T_out, T_kv]
    ref = logsumexp(np.where(seen[:, None], logits, -np.inf), axis=-1).transpose(0, 2, 1)
    np.testing.assert_allclose(oracle.xattn_lse(qc, pos, k, a, b, scale), ref, rtol=1e-12, atol=1e-12)


def test_xattn_lse_of_copies_at_every_position_is_the_full_causal_lse():
    """PT mode: copies of every base row, with the base rows' own q, see keys 0..t -- the
    base stream's lse with a window covering the whole sequence."""
    q, k, _, a, b = _rand_inputs(97, 2, 33, 4, 2, 16)
    pos = np.tile(np.arange(33, dtype=np.int32), (2, 1))
    np.testing.assert_allclose(oracle.xattn_lse(q, pos, k, a, b, 0.25), oracle.swa_lse(q, k, a, b, 33, 0.25),
                               rtol=1e-13, atol=1e-13)
