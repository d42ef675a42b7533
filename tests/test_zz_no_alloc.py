"""orthros_xattn_fwd_noalloc, called through the C ABI, against the workspace
entry point orthros_xattn_fwd on the same inputs.

The no-alloc variant exists for callers that cannot allocate device memory
(a plug-in whose host runtime owns all device memory, a latency-bound loop that
must never call cudaMalloc); its split-KV partials live in one fixed device
array inside the library.  Both entry points run the same kernels on the same
inputs, so their outputs must agree bit for bit; each is also held to the fp64
oracle.  Two calls in a row with different inputs check that the shared array's
leftover contents from the previous call never leak into a result.  This file is
collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import long_context_attention_orthros_gb300 as orth
import oracle
from synthetic import PrefillConfig, make_prefill
from tests.gpu_util import assert_parity, bf, bits, dev, f32, i32, val

NOALLOC_MAX_BYTES = 8 << 20  # ORTHROS_XATTN_NOALLOC_MAX_BYTES in include/orthros.h


def _entry():
    L = orth.lib()
    fn = L.orthros_xattn_fwd_noalloc
    P, I, F, L64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_int64
    fn.restype = I
    fn.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, F, L64, L64, L64, P, P]
    return fn


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _run(fn, cfg, seed, stream):
    inp = make_prefill(cfg, seed)
    k, v, qc, pos = bf(inp.k), bf(inp.v), bf(inp.qc_raw), i32(inp.pos)
    ac, bc = f32(inp.alpha_c), f32(inp.beta_c)
    ref = orth.xattn_fwd(qc, pos, k, v, ac, bc, scale=cfg.scale)
    out = torch.full_like(ref, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    st = fn(_p(qc), _p(pos), _p(k), _p(v), _p(ac), _p(bc), _p(out), cfg.B, cfg.T_out, cfg.T,
            cfg.Hq, cfg.Hkv, cfg.d, ctypes.c_float(cfg.scale), 0, 0, 0, _p(err), stream)
    assert st == 0, orth.lib().orthros_status_string(st)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return inp, ref, out


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls():
    fn = _entry()
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev()).cuda_stream)
    cases = [PrefillConfig("na1", B=2, T=5000, Hq=32, Hkv=8, d=128, T_out=1),
             PrefillConfig("na2", B=1, T=3001, Hq=8, Hkv=2, d=128, T_out=3, positions="shuffled")]
    for i, cfg in enumerate(cases):
        need = orth.xattn_workspace_size(cfg.B, cfg.T_out, cfg.T, cfg.Hq, cfg.Hkv, cfg.d)
        assert 256 < need <= NOALLOC_MAX_BYTES  # the split path that really uses the scratch
        inp, ref, out = _run(fn, cfg, 500 + i, stream)
        np.testing.assert_array_equal(bits(out), bits(ref), err_msg=f"no-alloc call {i + 1}")
        want = oracle.xattn(inp.qc_raw, inp.pos, inp.k, inp.v, inp.alpha_c, inp.beta_c, cfg.scale)
        assert_parity(val(out), want, f"no-alloc call {i + 1} vs oracle")


@pytest.mark.gpu
def test_noalloc_many_copies_take_the_kernel_without_partials():
    """T_out * G >= 256 runs on the tensor-memory kernel, which keeps no partials: the
    size query gives the 256-byte minimum however long the keys, and the no-alloc entry
    point serves it."""
    fn = _entry()
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev()).cuda_stream)
    cfg = PrefillConfig("na3", B=1, T=20000, Hq=8, Hkv=2, d=128, T_out=64, positions="shuffled")
    assert orth.xattn_workspace_size(cfg.B, cfg.T_out, cfg.T, cfg.Hq, cfg.Hkv, cfg.d) == 256
    inp, ref, out = _run(fn, cfg, 503, stream)
    np.testing.assert_array_equal(bits(out), bits(ref))
    want = oracle.xattn(inp.qc_raw, inp.pos, inp.k, inp.v, inp.alpha_c, inp.beta_c, cfg.scale)
    assert_parity(val(out), want, "no-alloc many copies vs oracle")


@pytest.mark.gpu
def test_noalloc_rejects_sizes_beyond_its_array():
    fn = _entry()
    B, T_out, T_kv, Hq, Hkv, d = 8, 4, 1 << 20, 32, 8, 128
    need = orth.xattn_workspace_size(B, T_out, T_kv, Hq, Hkv, d)
    assert need > NOALLOC_MAX_BYTES
    x = torch.zeros(16, dtype=torch.bfloat16, device=dev())
    st = fn(_p(x), _p(x), _p(x), _p(x), _p(x), _p(x), _p(x), B, T_out, T_kv, Hq, Hkv, d,
            ctypes.c_float(0.1), 0, 0, 0, None, None)
    assert st == 3  # ORTHROS_ERR_WORKSPACE, before anything is launched


def test_noalloc_statuses_match_the_workspace_entry_point():
    """Refused sizes give the status orthros_xattn_fwd gives (host checks only: no GPU)."""
    from long_context_attention_orthros_gb300 import build
    build.build()
    fn = _entry()
    L = orth.lib()
    buf = (ctypes.c_uint8 * 64)()
    p = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)
    P, I, F, L64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_int64, ctypes.c_size_t
    L.orthros_xattn_fwd.restype = I
    L.orthros_xattn_fwd.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, F, L64, L64, L64, P, SZ, P, P]
    for (B, T_out, T_kv, Hq, Hkv, d), want in (((1, 1, 64, 4, 2, 96), 2),  # head dimension
                                              ((1, 1, 64, 6, 4, 128), 2),  # grouping
                                              ((1, 1, 64, 96, 3, 128), 2),
                                              ((0, 1, 64, 4, 2, 128), 1),  # sizes
                                              ((1, -1, 64, 4, 2, 128), 1),
                                              ((1, 1, 0, 4, 2, 128), 1)):
        a = fn(p, p, p, p, p, p, p, B, T_out, T_kv, Hq, Hkv, d, ctypes.c_float(0.1), 0, 0, 0, None, None)
        b = L.orthros_xattn_fwd(p, p, p, p, p, p, p, B, T_out, T_kv, Hq, Hkv, d, ctypes.c_float(0.1), 0, 0, 0,
                                p, 64, None, None)
        assert a == b == want, (B, T_out, T_kv, Hq, Hkv, d, a, b)
