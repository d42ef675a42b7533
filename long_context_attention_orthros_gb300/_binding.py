"""ctypes binding of liborthros.so (the C ABI declared in include/orthros.h).

Only argument marshalling happens here: shapes and strides are read off torch
tensors, device pointers and the current CUDA stream are handed to the C entry
points, and a non-OK status becomes an exception.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "_lib", "liborthros.so")

DEVERR_POSITION = 1
DEVERR_CACHE_FULL = 2
DEVERR_TIMEOUT = 4
DEVERR_RANGE = 8

_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported configuration",
           3: "workspace missing or too small", 4: "CUDA error"}


class OrthrosError(RuntimeError):
    pass


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """Load liborthros.so (built by build.py / __graft_entry__.build()); raise if missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(library_path):
                raise OrthrosError(
                    f"{library_path} is missing: build it with "
                    "`python -m long_context_attention_orthros_gb300.build`")
            L = ctypes.CDLL(library_path)
            P, I, F, L64, SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_int64,
                                ctypes.c_size_t)
            L.orthros_status_string.restype = ctypes.c_char_p
            L.orthros_status_string.argtypes = [I]
            L.orthros_version.restype = I
            L.orthros_swa_fwd.restype = I
            L.orthros_swa_fwd.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, F, L64, L64, L64, P, P]
            L.orthros_swa_fwd_rows.restype = I
            L.orthros_swa_fwd_rows.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, F, L64, L64, L64, I, I, P, P]
            L.orthros_xattn_workspace_size.restype = SZ
            L.orthros_xattn_workspace_size.argtypes = [I, I, I, I, I, I]
            L.orthros_xattn_fwd.restype = I
            L.orthros_xattn_fwd.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, F, L64, L64, L64,
                                            P, SZ, P, P]
            L.orthros_prefill_workspace_size.restype = SZ
            L.orthros_prefill_workspace_size.argtypes = [I, I, I, I, I, I]
            L.orthros_prefill_fwd.restype = I
            L.orthros_prefill_fwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F,
                                              L64, L64, L64, L64, L64, P, SZ, P, P]
            L.orthros_decode_workspace_size.restype = SZ
            L.orthros_decode_workspace_size.argtypes = [I, I, I, I, I]
            L.orthros_decode_step.restype = I
            L.orthros_decode_step.argtypes = [P, P, P, P, P, P, P, I, P, P, P, P, P, P, I, I, I, I,
                                              I, F, P, SZ, P, P]
            L.orthros_swa_bwd_workspace_size.restype = SZ
            L.orthros_swa_bwd_workspace_size.argtypes = [I, I, I, I, I]
            L.orthros_swa_bwd.restype = I
            L.orthros_swa_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, P,
                                          SZ, P, P]
            L.orthros_swa_fwd_lse.restype = I
            L.orthros_swa_fwd_lse.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, F, L64, L64, L64, P, P]
            L.orthros_xattn_bwd_workspace_size.restype = SZ
            L.orthros_xattn_bwd_workspace_size.argtypes = [I, I, I, I, I, I]
            L.orthros_xattn_bwd.restype = I
            L.orthros_xattn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F,
                                            I, P, SZ, P, P]
            L.orthros_attn_bwd_workspace_size.restype = SZ
            L.orthros_attn_bwd_workspace_size.argtypes = [I, I, I, I, I, I]
            L.orthros_attn_bwd.restype = I
            L.orthros_attn_bwd.argtypes = [P] * 23 + [I, I, I, I, I, I, I, F, P, SZ, P, P]
            L.orthros_xattn_fwd_lse.restype = I
            L.orthros_xattn_fwd_lse.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, L64, L64, L64,
                                                P, SZ, P, P]
            _lib = L
    return _lib


def _check(status: int, what: str) -> None:
    if status != 0:
        raise OrthrosError(f"{what}: {_STATUS.get(status, status)}")


def _ptr(t):
    """Device pointer of a tensor argument.  Every pointer the library takes is a device
    pointer of the call's GPU (the current device inside the calls below): a host tensor or
    one on another GPU is refused here rather than handed to a kernel."""
    if t is None:
        return None
    if not t.is_cuda or t.device.index != torch.cuda.current_device():
        raise OrthrosError(f"tensor arguments must be CUDA tensors on the call's device (got {t.device})")
    return ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _bf16_rows(t: torch.Tensor, name: str) -> int:
    """Check a [B, T, H, d] bf16 CUDA tensor whose (T, H, d) block is dense; return its batch stride."""
    if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 4:
        raise OrthrosError(f"{name} must be a 4-D bf16 CUDA tensor [B, T, H, d]")
    B, T, H, d = t.shape
    # strides of size-1 dimensions are irrelevant (numpy/torch may report anything there)
    if ((d > 1 and t.stride(3) != 1) or (H > 1 and t.stride(2) != d)
            or (T > 1 and t.stride(1) != H * d)):
        raise OrthrosError(f"{name}: the [T, H, d] part must be dense (d contiguous)")
    return t.stride(0) if B > 1 else T * H * d


def _vec(t: torch.Tensor, name: str, Hq: int, d: int) -> None:
    if t.dtype != torch.float32 or not t.is_cuda or tuple(t.shape) != (Hq, d) or not t.is_contiguous():
        raise OrthrosError(f"{name} must be a contiguous fp32 CUDA tensor [Hq, d]")


def _scale(scale, d):
    return 1.0 / math.sqrt(d) if scale is None else float(scale)


def swa_fwd(q_raw, k, v, alpha, beta, window: int = 128, scale=None, out=None, dev_err=None):
    """Eq. (4): o[b, t] = softmax over keys max(0, t-window+1)..t of (q . k) * scale, applied to v,
    with q = q_raw * alpha + beta.  q_raw [B, Tq, Hq, d] (Tq >= T, only the first T rows are
    read, so copies may be appended after the base tokens); k, v [B, T, Hkv, d]."""
    B, T, Hkv, d = k.shape
    Hq = q_raw.shape[2]
    qs = _bf16_rows(q_raw, "q_raw")
    ks = _bf16_rows(k, "k")
    if _bf16_rows(v, "v") != ks or v.shape != k.shape:
        raise OrthrosError("k and v must have the same shape and strides")
    if q_raw.shape[0] != B or q_raw.shape[1] < T or q_raw.shape[3] != d:
        raise OrthrosError("q_raw shape does not match k")
    _vec(alpha, "alpha", Hq, d)
    _vec(beta, "beta", Hq, d)
    if out is None:
        out = torch.empty((B, T, Hq, d), dtype=torch.bfloat16, device=k.device)
    os_ = _bf16_rows(out, "out")
    with torch.cuda.device(k.device):
        st = lib().orthros_swa_fwd(_ptr(q_raw), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(out),
                                   B, T, Hq, Hkv, d, int(window), _scale(scale, d), qs, ks, os_,
                                   _ptr(dev_err), _stream(k.device))
    _check(st, "orthros_swa_fwd")
    return out


def swa_fwd_rows(q_raw, k, v, alpha, beta, row_begin: int, row_end: int, window: int = 128, scale=None,
                 out=None, dev_err=None):
    """swa_fwd for output rows row_begin..row_end-1 of every sequence only (chunked prefill);
    other rows of `out` are left as they are.  row_begin a multiple of 128, row_end a multiple
    of 128 or T.  Keys are read from row max(0, row_begin - window + 1)."""
    B, T, Hkv, d = k.shape
    Hq = q_raw.shape[2]
    qs = _bf16_rows(q_raw, "q_raw")
    ks = _bf16_rows(k, "k")
    if _bf16_rows(v, "v") != ks or v.shape != k.shape:
        raise OrthrosError("k and v must have the same shape and strides")
    if q_raw.shape[0] != B or q_raw.shape[1] < T or q_raw.shape[3] != d:
        raise OrthrosError("q_raw shape does not match k")
    _vec(alpha, "alpha", Hq, d)
    _vec(beta, "beta", Hq, d)
    if out is None:
        out = torch.empty((B, T, Hq, d), dtype=torch.bfloat16, device=k.device)
    os_ = _bf16_rows(out, "out")
    with torch.cuda.device(k.device):
        st = lib().orthros_swa_fwd_rows(_ptr(q_raw), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(out),
                                        B, T, Hq, Hkv, d, int(window), _scale(scale, d), qs, ks, os_,
                                        int(row_begin), int(row_end), _ptr(dev_err), _stream(k.device))
    _check(st, "orthros_swa_fwd_rows")
    return out


def xattn_workspace_size(B, T_out, T_kv, Hq, Hkv, d) -> int:
    return int(lib().orthros_xattn_workspace_size(B, T_out, T_kv, Hq, Hkv, d))


def decode_workspace_size(B, L_max, Hq, Hkv, d) -> int:
    return int(lib().orthros_decode_workspace_size(B, L_max, Hq, Hkv, d))


def xattn_fwd(qc_raw, pos, k, v, alpha_c, beta_c, scale=None, out=None, workspace=None, dev_err=None,
              lse=None):
    """Eq. (5): copy i of sequence b at original position pos[b, i] attends over k/v rows
    0..pos[b, i].  qc_raw [B, T_out, Hq, d] (may be a view of an appended buffer);
    pos int32 [B, T_out]; k, v [B, T_kv, Hkv, d].  With lse (fp32 [B, T_out, Hq], or True for
    a fresh one) each copy row's log-sum-exp is written too, for xattn_bwd, and (out, lse)
    is returned."""
    B, T_kv, Hkv, d = k.shape
    T_out, Hq = qc_raw.shape[1], qc_raw.shape[2]
    qs = _bf16_rows(qc_raw, "qc_raw")
    ks = _bf16_rows(k, "k")
    if _bf16_rows(v, "v") != ks or v.shape != k.shape:
        raise OrthrosError("k and v must have the same shape and strides")
    if pos.dtype != torch.int32 or tuple(pos.shape) != (B, T_out) or not pos.is_contiguous():
        raise OrthrosError("pos must be a contiguous int32 tensor [B, T_out]")
    _vec(alpha_c, "alpha_c", Hq, d)
    _vec(beta_c, "beta_c", Hq, d)
    if out is None:
        out = torch.empty((B, T_out, Hq, d), dtype=torch.bfloat16, device=k.device)
    os_ = _bf16_rows(out, "out")
    need = xattn_workspace_size(B, T_out, T_kv, Hq, Hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=k.device)
    if lse is True:
        lse = torch.empty((B, T_out, Hq), dtype=torch.float32, device=k.device)
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (B, T_out, Hq) or
                            not lse.is_contiguous()):
        raise OrthrosError("lse must be a contiguous fp32 tensor [B, T_out, Hq]")
    with torch.cuda.device(k.device):
        if lse is None:
            st = lib().orthros_xattn_fwd(_ptr(qc_raw), _ptr(pos), _ptr(k), _ptr(v), _ptr(alpha_c),
                                         _ptr(beta_c), _ptr(out), B, T_out, T_kv, Hq, Hkv, d,
                                         _scale(scale, d), qs, ks, os_, _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), _ptr(dev_err),
                                         _stream(k.device))
        else:
            st = lib().orthros_xattn_fwd_lse(_ptr(qc_raw), _ptr(pos), _ptr(k), _ptr(v), _ptr(alpha_c),
                                             _ptr(beta_c), _ptr(out), _ptr(lse), B, T_out, T_kv, Hq, Hkv, d,
                                             _scale(scale, d), qs, ks, os_, _ptr(workspace),
                                             workspace.numel() * workspace.element_size(), _ptr(dev_err),
                                             _stream(k.device))
    _check(st, "orthros_xattn_fwd")
    return out if lse is None else (out, lse)


def prefill_workspace_size(B, T, T_out, Hq, Hkv, d) -> int:
    return int(lib().orthros_prefill_workspace_size(B, T, T_out, Hq, Hkv, d))


def prefill_fwd(q_raw, k, v, alpha, beta, qc_raw, pos, alpha_c, beta_c, window: int = 128, scale=None,
                out=None, out_c=None, workspace=None, dev_err=None):
    """One prefill layer in one call: swa_fwd for the base stream, then xattn_fwd (T_kv = T)
    for the output copies.  Returns (o, oc)."""
    B, T, Hkv, d = k.shape
    Hq = q_raw.shape[2]
    T_out = qc_raw.shape[1]
    qs = _bf16_rows(q_raw, "q_raw")
    qcs = _bf16_rows(qc_raw, "qc_raw")
    ks = _bf16_rows(k, "k")
    if _bf16_rows(v, "v") != ks or v.shape != k.shape:
        raise OrthrosError("k and v must have the same shape and strides")
    if q_raw.shape[0] != B or q_raw.shape[1] < T or q_raw.shape[3] != d:
        raise OrthrosError("q_raw shape does not match k")
    if qc_raw.shape[0] != B or qc_raw.shape[2] != Hq or qc_raw.shape[3] != d:
        raise OrthrosError("qc_raw shape does not match q_raw")
    if pos.dtype != torch.int32 or tuple(pos.shape) != (B, T_out) or not pos.is_contiguous():
        raise OrthrosError("pos must be a contiguous int32 tensor [B, T_out]")
    for t, nm in ((alpha, "alpha"), (beta, "beta"), (alpha_c, "alpha_c"), (beta_c, "beta_c")):
        _vec(t, nm, Hq, d)
    if out is None:
        out = torch.empty((B, T, Hq, d), dtype=torch.bfloat16, device=k.device)
    if out_c is None:
        out_c = torch.empty((B, T_out, Hq, d), dtype=torch.bfloat16, device=k.device)
    os_ = _bf16_rows(out, "out")
    ocs = _bf16_rows(out_c, "out_c")
    if workspace is None:
        workspace = torch.empty(max(prefill_workspace_size(B, T, T_out, Hq, Hkv, d), 256),
                                dtype=torch.uint8, device=k.device)
    with torch.cuda.device(k.device):
        st = lib().orthros_prefill_fwd(_ptr(q_raw), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(out),
                                       _ptr(qc_raw), _ptr(pos), _ptr(alpha_c), _ptr(beta_c), _ptr(out_c),
                                       B, T, T_out, Hq, Hkv, d, int(window), _scale(scale, d), qs, ks, os_,
                                       qcs, ocs, _ptr(workspace), workspace.numel() * workspace.element_size(),
                                       _ptr(dev_err), _stream(k.device))
    _check(st, "orthros_prefill_fwd")
    return out, out_c


def swa_bwd_workspace_size(B, T, Hq, Hkv, d) -> int:
    return int(lib().orthros_swa_bwd_workspace_size(B, T, Hq, Hkv, d))


def swa_fwd_lse(q_raw, k, v, alpha, beta, window: int = 128, scale=None, out=None, lse=None, dev_err=None):
    """swa_fwd that also returns each row's log-sum-exp, fp32 [B, T, Hq] (natural log of the
    softmax normaliser), for swa_bwd.  Returns (o, lse)."""
    B, T, Hkv, d = k.shape
    Hq = q_raw.shape[2]
    qs = _bf16_rows(q_raw, "q_raw")
    ks = _bf16_rows(k, "k")
    if _bf16_rows(v, "v") != ks or v.shape != k.shape:
        raise OrthrosError("k and v must have the same shape and strides")
    if q_raw.shape[0] != B or q_raw.shape[1] < T or q_raw.shape[3] != d:
        raise OrthrosError("q_raw shape does not match k")
    _vec(alpha, "alpha", Hq, d)
    _vec(beta, "beta", Hq, d)
    if out is None:
        out = torch.empty((B, T, Hq, d), dtype=torch.bfloat16, device=k.device)
    if lse is None:
        lse = torch.empty((B, T, Hq), dtype=torch.float32, device=k.device)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, T, Hq) or not lse.is_contiguous():
        raise OrthrosError("lse must be a contiguous fp32 tensor [B, T, Hq]")
    os_ = _bf16_rows(out, "out")
    with torch.cuda.device(k.device):
        st = lib().orthros_swa_fwd_lse(_ptr(q_raw), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(out), _ptr(lse),
                                       B, T, Hq, Hkv, d, int(window), _scale(scale, d), qs, ks, os_, _ptr(dev_err),
                                       _stream(k.device))
    _check(st, "orthros_swa_fwd_lse")
    return out, lse


def swa_bwd(q_raw, k, v, alpha, beta, o, dO, window: int = 128, scale=None, workspace=None, dev_err=None,
            lse=None):
    """Gradient of Eq. (4) with its scale-offset: returns fp32 (dq_raw, dk, dv, dalpha, dbeta) for
    the output gradient dO, given the forward inputs and the forward output o.  q_raw, o, dO
    [B, T, Hq, d] and k, v [B, T, Hkv, d], all dense bf16; alpha, beta [Hq, d] fp32."""
    B, T, Hkv, d = k.shape
    Hq = q_raw.shape[2]
    for t, nm, shp in ((q_raw, "q_raw", (B, T, Hq, d)), (o, "o", (B, T, Hq, d)), (dO, "dO", (B, T, Hq, d)),
                       (k, "k", (B, T, Hkv, d)), (v, "v", (B, T, Hkv, d))):
        if t.dtype != torch.bfloat16 or not t.is_cuda or tuple(t.shape) != shp or not t.is_contiguous():
            raise OrthrosError(f"{nm} must be a contiguous bf16 CUDA tensor {shp}")
    _vec(alpha, "alpha", Hq, d)
    _vec(beta, "beta", Hq, d)
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (B, T, Hq) or not lse.is_contiguous()):
        raise OrthrosError("lse must be a contiguous fp32 tensor [B, T, Hq] (from swa_fwd_lse)")
    f32 = dict(dtype=torch.float32, device=k.device)
    dq = torch.empty((B, T, Hq, d), **f32)
    dk = torch.empty((B, T, Hkv, d), **f32)
    dv = torch.empty((B, T, Hkv, d), **f32)
    dalpha = torch.empty((Hq, d), **f32)
    dbeta = torch.empty((Hq, d), **f32)
    if workspace is None:
        workspace = torch.empty(max(swa_bwd_workspace_size(B, T, Hq, Hkv, d), 256), dtype=torch.uint8,
                                device=k.device)
    with torch.cuda.device(k.device):
        st = lib().orthros_swa_bwd(_ptr(q_raw), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(o), _ptr(dO),
                                   _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dalpha), _ptr(dbeta), B, T, Hq, Hkv, d,
                                   int(window), _scale(scale, d), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _ptr(dev_err), _stream(k.device))
    _check(st, "orthros_swa_bwd")
    return dq, dk, dv, dalpha, dbeta


def xattn_bwd_workspace_size(B, T_out, T_kv, Hq, Hkv, d) -> int:
    return int(lib().orthros_xattn_bwd_workspace_size(B, T_out, T_kv, Hq, Hkv, d))


def xattn_bwd(qc_raw, pos, k, v, alpha_c, beta_c, oc, dOc, scale=None, dk=None, dv=None, workspace=None,
              dev_err=None, lse=None):
    """Gradient of Eq. (5) with the copies' scale-offset: returns fp32 (dqc_raw, dk, dv, dalpha_c,
    dbeta_c).  Passing dk, dv (fp32 [B, T_kv, Hkv, d], e.g. from swa_bwd) adds the copies' share
    to them in place; otherwise fresh tensors hold the copies' share alone.  qc_raw, oc, dOc
    [B, T_out, Hq, d] and k, v [B, T_kv, Hkv, d] dense bf16; pos int32 [B, T_out]; lse (optional)
    the forward's fp32 [B, T_out, Hq] log-sum-exp (xattn_fwd with lse)."""
    B, T_kv, Hkv, d = k.shape
    T_out, Hq = qc_raw.shape[1], qc_raw.shape[2]
    for t, nm, shp in ((qc_raw, "qc_raw", (B, T_out, Hq, d)), (oc, "oc", (B, T_out, Hq, d)),
                       (dOc, "dOc", (B, T_out, Hq, d)), (k, "k", (B, T_kv, Hkv, d)), (v, "v", (B, T_kv, Hkv, d))):
        if t.dtype != torch.bfloat16 or not t.is_cuda or tuple(t.shape) != shp or not t.is_contiguous():
            raise OrthrosError(f"{nm} must be a contiguous bf16 CUDA tensor {shp}")
    if pos.dtype != torch.int32 or tuple(pos.shape) != (B, T_out) or not pos.is_contiguous():
        raise OrthrosError("pos must be a contiguous int32 tensor [B, T_out]")
    _vec(alpha_c, "alpha_c", Hq, d)
    _vec(beta_c, "beta_c", Hq, d)
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (B, T_out, Hq) or
                            not lse.is_contiguous()):
        raise OrthrosError("lse must be a contiguous fp32 tensor [B, T_out, Hq]")
    f32 = dict(dtype=torch.float32, device=k.device)
    accumulate = dk is not None
    if (dk is None) != (dv is None):
        raise OrthrosError("pass both dk and dv, or neither")
    for t, nm in ((dk, "dk"), (dv, "dv")):
        if t is not None and (t.dtype != torch.float32 or tuple(t.shape) != (B, T_kv, Hkv, d)
                              or not t.is_contiguous()):
            raise OrthrosError(f"{nm} must be a contiguous fp32 tensor [B, T_kv, Hkv, d]")
    if not accumulate:
        dk = torch.empty((B, T_kv, Hkv, d), **f32)
        dv = torch.empty((B, T_kv, Hkv, d), **f32)
    dq = torch.empty((B, T_out, Hq, d), **f32)
    dalpha = torch.empty((Hq, d), **f32)
    dbeta = torch.empty((Hq, d), **f32)
    if workspace is None:
        workspace = torch.empty(max(xattn_bwd_workspace_size(B, T_out, T_kv, Hq, Hkv, d), 256), dtype=torch.uint8,
                                device=k.device)
    with torch.cuda.device(k.device):
        st = lib().orthros_xattn_bwd(_ptr(qc_raw), _ptr(pos), _ptr(k), _ptr(v), _ptr(alpha_c), _ptr(beta_c),
                                     _ptr(oc), _ptr(dOc), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dalpha),
                                     _ptr(dbeta),
                                     B, T_out, T_kv, Hq, Hkv, d, _scale(scale, d), int(accumulate),
                                     _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     _ptr(dev_err), _stream(k.device))
    _check(st, "orthros_xattn_bwd")
    return dq, dk, dv, dalpha, dbeta


def attn_bwd_workspace_size(B, T, T_out, Hq, Hkv, d) -> int:
    return int(lib().orthros_attn_bwd_workspace_size(B, T, T_out, Hq, Hkv, d))


def attn_bwd(q_raw, k, v, alpha, beta, o, dO, qc_raw, pos, alpha_c, beta_c, oc, dOc, window: int = 128,
             scale=None, lse=None, lsec=None, workspace=None, dev_err=None):
    """A layer's attention gradient, both streams in one call: returns fp32 (dq_raw, dk, dv, dalpha,
    dbeta, dqc_raw, dalpha_c, dbeta_c), dk and dv holding both streams' shares.  Base tensors as
    swa_bwd, copy tensors as xattn_bwd (T_kv = T); lse / lsec the forwards' log-sum-exp or None."""
    B, T, Hkv, d = k.shape
    Hq, T_out = q_raw.shape[2], qc_raw.shape[1]
    for t, nm, shp in ((q_raw, "q_raw", (B, T, Hq, d)), (o, "o", (B, T, Hq, d)), (dO, "dO", (B, T, Hq, d)),
                       (qc_raw, "qc_raw", (B, T_out, Hq, d)), (oc, "oc", (B, T_out, Hq, d)),
                       (dOc, "dOc", (B, T_out, Hq, d)), (k, "k", (B, T, Hkv, d)), (v, "v", (B, T, Hkv, d))):
        if t.dtype != torch.bfloat16 or not t.is_cuda or tuple(t.shape) != shp or not t.is_contiguous():
            raise OrthrosError(f"{nm} must be a contiguous bf16 CUDA tensor {shp}")
    if pos.dtype != torch.int32 or tuple(pos.shape) != (B, T_out) or not pos.is_contiguous():
        raise OrthrosError("pos must be a contiguous int32 tensor [B, T_out]")
    for t, nm in ((alpha, "alpha"), (beta, "beta"), (alpha_c, "alpha_c"), (beta_c, "beta_c")):
        _vec(t, nm, Hq, d)
    for t, nm, shp in ((lse, "lse", (B, T, Hq)), (lsec, "lsec", (B, T_out, Hq))):
        if t is not None and (t.dtype != torch.float32 or tuple(t.shape) != shp or not t.is_contiguous()):
            raise OrthrosError(f"{nm} must be a contiguous fp32 tensor {shp}")
    f32 = dict(dtype=torch.float32, device=k.device)
    out = [torch.empty(shp, **f32) for shp in ((B, T, Hq, d), (B, T, Hkv, d), (B, T, Hkv, d), (Hq, d), (Hq, d),
                                                (B, T_out, Hq, d), (Hq, d), (Hq, d))]
    if workspace is None:
        workspace = torch.empty(attn_bwd_workspace_size(B, T, T_out, Hq, Hkv, d), dtype=torch.uint8,
                                device=k.device)
    with torch.cuda.device(k.device):
        st = lib().orthros_attn_bwd(_ptr(q_raw), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(o), _ptr(dO),
                                    _ptr(lse), _ptr(qc_raw), _ptr(pos), _ptr(alpha_c), _ptr(beta_c), _ptr(oc),
                                    _ptr(dOc), _ptr(lsec), *[_ptr(t) for t in out], B, T, T_out, Hq, Hkv, d,
                                    int(window), _scale(scale, d), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _ptr(dev_err),
                                    _stream(k.device))
    _check(st, "orthros_attn_bwd")
    return tuple(out)


def decode_workspace(B, L_max, Hq, Hkv, d, device) -> torch.Tensor:
    """A zero-filled workspace for decode_step (reusable step after step)."""
    return torch.zeros(max(decode_workspace_size(B, L_max, Hq, Hkv, d), 256), dtype=torch.uint8,
                       device=device)


def decode_step(q_new, qc_new, k_new, v_new, k_cache, v_cache, cache_len, alpha, beta, alpha_c,
                beta_c, window: int = 128, scale=None, o=None, oc=None, workspace=None, dev_err=None):
    """One decode step: append k_new/v_new at row cache_len[b], base SWA for q_new, full-cache
    attention for the copy qc_new, then cache_len += 1.  q_new, qc_new [B, Hq, d];
    k_new, v_new [B, Hkv, d]; k_cache, v_cache [B, L_max, Hkv, d]; cache_len int32 [B]."""
    B, L_max, Hkv, d = k_cache.shape
    Hq = q_new.shape[1]
    for t, nm, shp in ((q_new, "q_new", (B, Hq, d)), (qc_new, "qc_new", (B, Hq, d)),
                       (k_new, "k_new", (B, Hkv, d)), (v_new, "v_new", (B, Hkv, d)),
                       (k_cache, "k_cache", (B, L_max, Hkv, d)), (v_cache, "v_cache", (B, L_max, Hkv, d))):
        if t.dtype != torch.bfloat16 or not t.is_cuda or tuple(t.shape) != shp or not t.is_contiguous():
            raise OrthrosError(f"{nm} must be a contiguous bf16 CUDA tensor {shp}")
    if cache_len.dtype != torch.int32 or tuple(cache_len.shape) != (B,) or not cache_len.is_cuda:
        raise OrthrosError("cache_len must be an int32 CUDA tensor [B]")
    for t, nm in ((alpha, "alpha"), (beta, "beta"), (alpha_c, "alpha_c"), (beta_c, "beta_c")):
        _vec(t, nm, Hq, d)
    if o is None:
        o = torch.empty((B, Hq, d), dtype=torch.bfloat16, device=k_cache.device)
    if oc is None:
        oc = torch.empty((B, Hq, d), dtype=torch.bfloat16, device=k_cache.device)
    if workspace is None:
        workspace = decode_workspace(B, L_max, Hq, Hkv, d, k_cache.device)
    with torch.cuda.device(k_cache.device):
        st = lib().orthros_decode_step(_ptr(q_new), _ptr(qc_new), _ptr(k_new), _ptr(v_new),
                                       _ptr(k_cache), _ptr(v_cache), _ptr(cache_len), L_max,
                                       _ptr(alpha), _ptr(beta), _ptr(alpha_c), _ptr(beta_c),
                                       _ptr(o), _ptr(oc), B, Hq, Hkv, d, int(window), _scale(scale, d),
                                       _ptr(workspace), workspace.numel() * workspace.element_size(),
                                       _ptr(dev_err), _stream(k_cache.device))
    _check(st, "orthros_decode_step")
    return o, oc
