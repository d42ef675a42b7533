"""GPU parity of the forward's per-row log-sum-exp (orthros_swa_fwd_lse) against the fp64
oracle, and of the gradient that takes it (orthros_swa_bwd with lse: the persistent
tensor-memory dq kernel) against the oracle's gradient.

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
