"""GPU parity of the base-stream gradient (orthros_swa_bwd: Eq. (4) with its
scale-offset) against the fp64 oracle's swa_bwd on the same seeded inputs.

The kernels multiply bf16 operands with fp32 accumulation: P and dS are rounded
to bf16 (unit roundoff u = 2**-8) before they meet dO, K and q; q enters dK
rounded once to bf16; D = dO . o uses the bf16 forward output.  Each rounding
perturbs a term by at most u relative and the perturbations of a sum are
independent, so the normwise relative error of every gradient stays a small
multiple of u / sqrt(3) ~ 2.3e-3.  The bar, per gradient tensor:
  ||got - ref||_2 <= 1e-2 * ||ref||_2            (about 2.5 u)
  max |got - ref| <= 3e-2 * max |ref|            (no element far off)
A masking or indexing mistake moves single elements by the size of the element
and fails the second bound; a dropped scale or term fails both."""
import math

import numpy as np
import pytest
import torch

import long_context_attention_orthros_gb300 as orth
import oracle
from synthetic import bf16_to_f32, normal_bf16, scale_offset
from tests.gpu_util import bf, dev, f32

pytestmark = pytest.mark.gpu

NORM_REL = 1e-2
MAX_REL = 3e-2
ZERO_ABS = 1e-4
NAMES = ("dq_raw", "dk", "dv", "dalpha", "dbeta")


def _inputs(seed, B, T, Hq, Hkv, d):
    q = normal_bf16(seed, "q_raw", (B, T, Hq, d))
    k = normal_bf16(seed, "k", (B, T, Hkv, d))
    v = normal_bf16(seed, "v", (B, T, Hkv, d))
    dO = normal_bf16(seed, "dO", (B, T, Hq, d))
    a, b = scale_offset(seed, Hq, d)
    return q, k, v, a, b, dO


def _gpu_grads(q, k, v, a, b, dO, w, scale):
    qg, kg, vg, dOg = bf(q), bf(k), bf(v), bf(dO)
    ag, bg = f32(a), f32(b)
    o = orth.swa_fwd(qg, kg, vg, ag, bg, window=w, scale=scale)
    got = orth.swa_bwd(qg, kg, vg, ag, bg, o, dOg, window=w, scale=scale)
    torch.cuda.synchronize()
    return [t.cpu().numpy().astype(np.float64) for t in got]


def _assert_grad(g, r, what):
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite"
    rn = float(np.linalg.norm(r))
    en = float(np.linalg.norm(g - r))
    mx = float(np.abs(g - r).max()) if g.size else 0.0
    rm = float(np.abs(r).max()) if r.size else 0.0
    if rn == 0.0:
        # exact zeros (w = 1: ds = dp - D with dp = D) come out as the fp32 cancellation of
        # dO . v taken in two summation orders: ~ sqrt(d) * 2**-24 * |dO| |v| ~ 1e-5 here
        assert mx <= ZERO_ABS, f"{what}: expected zeros, max |got| {mx:.3e}"
        return
    assert en <= NORM_REL * rn and mx <= MAX_REL * rm, (
        f"{what}: normwise {en / rn:.3e} (bar {NORM_REL}), max {mx:.3e} vs max|ref| {rm:.3e}")


@pytest.mark.parametrize("B,T,Hq,Hkv,d,w", [
    (1, 300, 8, 2, 128, 128),    # G=4, several dq tiles and dk/dv key blocks
    (2, 257, 16, 2, 128, 128),   # G=8 (the 8B-class grouping), ragged tail
    (1, 200, 4, 4, 64, 128),     # G=1, d=64
    (1, 190, 16, 1, 64, 33),     # G=16, narrow odd window
    (1, 150, 8, 4, 128, 1),      # w=1: o = v, no gradient in q, k, alpha, beta
    (1, 100, 4, 2, 128, 300),    # w >= T: full causal
    (1, 1200, 8, 2, 128, 1000),  # a window of many streamed key blocks
    (1, 5, 4, 1, 128, 128),      # T smaller than every tile
])
def test_swa_bwd_parity(B, T, Hq, Hkv, d, w):
    q, k, v, a, b, dO = _inputs(3000 + T, B, T, Hq, Hkv, d)
    scale = 1.0 / math.sqrt(d)
    got = _gpu_grads(q, k, v, a, b, dO, w, scale)
    ref = oracle.swa_bwd(q, k, v, a, b, dO, w, scale)
    for name, g, r in zip(NAMES, got, ref):
        _assert_grad(g, r, name)


def _slice_grads(q, k, v, a, b, dO, w, scale, lo, hi):
    """Oracle gradient of tokens lo..hi-1 alone (a sequence cut out of the long one)."""
    s = slice(lo, hi)
    return oracle.swa_bwd(np.ascontiguousarray(q[:, s]), np.ascontiguousarray(k[:, s]),
                          np.ascontiguousarray(v[:, s]), a, b, np.ascontiguousarray(dO[:, s]), w, scale)


def test_swa_bwd_training_size_sampled():
    """One 16K-token training sequence with 8B-class heads (32 query / 8 KV heads, d=128,
    w=128).  Row t's dq depends only on tokens t-w+1..t, and key j's dk, dv only on
    tokens j-w+1..j+w-1, so the oracle run on such a slice gives them exactly; a sample
    of rows and keys spread over the sequence (first, last, tile edges) is checked that
    way.  dalpha and dbeta are checked as the sums they are, over the GPU's own dq."""
    B, T, Hq, Hkv, d, w = 1, 16384, 32, 8, 128, 128
    q, k, v, a, b, dO = _inputs(4242, B, T, Hq, Hkv, d)
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv, da, db = _gpu_grads(q, k, v, a, b, dO, w, scale)
    for t in (0, 1, 127, 128, 4095, 8191, 8192, 12345, T - 2, T - 1):
        lo = max(0, t - w + 1)
        r = _slice_grads(q, k, v, a, b, dO, w, scale, lo, t + 1)
        _assert_grad(dq[:, t], r[0][:, t - lo], f"dq_raw row {t}")
    for j in (0, 63, 64, 5000, 9999, T - 129, T - 65, T - 1):
        lo, hi = max(0, j - w + 1), min(T, j + w)
        r = _slice_grads(q, k, v, a, b, dO, w, scale, lo, hi)
        _assert_grad(dk[:, j], r[1][:, j - lo], f"dk key {j}")
        _assert_grad(dv[:, j], r[2][:, j - lo], f"dv key {j}")
    dq_post = dq / a.astype(np.float64)  # dq = dq_raw / alpha (alpha ~ 1 +- 0.3)
    x = bf16_to_f32(q).astype(np.float64)
    _assert_grad(db, dq_post.sum(axis=(0, 1)), "dbeta as the sum of dq")
    _assert_grad(da, (x * dq_post).sum(axis=(0, 1)), "dalpha as the sum of x * dq")


def test_swa_bwd_is_deterministic_in_dq_dk_dv():
    """dq, dk and dv are each written by one thread (no atomics): two calls agree bit for bit."""
    B, T, Hq, Hkv, d, w = 1, 700, 16, 2, 128, 128
    q, k, v, a, b, dO = _inputs(55, B, T, Hq, Hkv, d)
    qg, kg, vg, dOg, ag, bg = bf(q), bf(k), bf(v), bf(dO), f32(a), f32(b)
    o = orth.swa_fwd(qg, kg, vg, ag, bg, window=w)
    g1 = orth.swa_bwd(qg, kg, vg, ag, bg, o, dOg, window=w)
    g2 = orth.swa_bwd(qg, kg, vg, ag, bg, o, dOg, window=w)
    torch.cuda.synchronize()
    for t1, t2 in zip(g1[:3], g2[:3]):
        assert torch.equal(t1, t2)
