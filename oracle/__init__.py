"""fp64 CPU oracle for the Orthros per-layer attention operator.

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline / reference arm are the only users.  The product path
(the CUDA library and its binding) never imports this package.

The arithmetic lives in ``orthros_oracle.c`` (plain C, double precision); this
module compiles it with gcc on first use (or via :func:`build`) and wraps it
with numpy marshalling.  Inputs are the bf16 bit patterns (``numpy.uint16``) and
fp32 vectors that ``synthetic.py`` produces.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "orthros_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liborthros_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library (gcc, OpenMP, no FP contraction)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            lib.oracle_num_threads.restype = I
            lib.oracle_set_num_threads.argtypes = [I]
            lib.oracle_set_num_threads.restype = None
            lib.oracle_swa.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, D]
            lib.oracle_swa_rows.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, D, P, P, I]
            lib.oracle_xattn.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, D]
            lib.oracle_swa_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, D]
            lib.oracle_xattn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, D]
            lib.oracle_swa_lse.argtypes = [P, P, P, P, P, I, I, I, I, I, I, D]
            lib.oracle_xattn_lse.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, D]
            lib.oracle_decode_step.argtypes = [P, P, P, P, P, P, P, I, P, P, P, P, P, P,
                                               I, I, I, I, I, D]
            for f in (lib.oracle_swa, lib.oracle_swa_rows, lib.oracle_xattn, lib.oracle_decode_step,
                      lib.oracle_swa_bwd, lib.oracle_xattn_bwd, lib.oracle_swa_lse, lib.oracle_xattn_lse):
                f.restype = I
            _lib = lib
    return _lib


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    """Threads of later oracle calls from this thread (timing only; the values do not depend
    on it)."""
    _load().oracle_set_num_threads(int(n))


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid argument (rc={rc})")


def swa(q_raw, k, v, alpha, beta, window: int, scale: float) -> np.ndarray:
    """Eq. (4) at every base position.  q_raw [B,T,Hq,d], k/v [B,T,Hkv,d] bf16 bits."""
    B, T, Hq, d = q_raw.shape
    Hkv = k.shape[2]
    assert k.shape == v.shape == (B, T, Hkv, d)
    q_raw, pq = _c(q_raw, np.uint16)
    k, pk = _c(k, np.uint16)
    v, pv = _c(v, np.uint16)
    alpha, pa = _c(alpha, np.float32)
    beta, pb = _c(beta, np.float32)
    o = np.zeros((B, T, Hq, d), np.float64)
    rc = _load().oracle_swa(pq, pk, pv, pa, pb, o.ctypes.data_as(ctypes.c_void_p),
                            B, T, Hq, Hkv, d, int(window), float(scale))
    _check(rc, "swa")
    return o


def swa_bwd(q_raw, k, v, alpha, beta, dO, window: int, scale: float):
    """Gradient of Eq. (4) with its scale-offset for an output gradient dO (bf16 bits
    [B,T,Hq,d]): returns fp64 (dq_raw [B,T,Hq,d], dk, dv [B,T,Hkv,d], dalpha, dbeta [Hq,d])."""
    B, T, Hq, d = q_raw.shape
    Hkv = k.shape[2]
    assert k.shape == v.shape == (B, T, Hkv, d) and dO.shape == q_raw.shape
    q_raw, pq = _c(q_raw, np.uint16)
    k, pk = _c(k, np.uint16)
    v, pv = _c(v, np.uint16)
    alpha, pa = _c(alpha, np.float32)
    beta, pb = _c(beta, np.float32)
    dO, pg = _c(dO, np.uint16)
    out = [np.zeros(s, np.float64) for s in ((B, T, Hq, d), (B, T, Hkv, d), (B, T, Hkv, d), (Hq, d), (Hq, d))]
    rc = _load().oracle_swa_bwd(pq, pk, pv, pa, pb, pg, *[o.ctypes.data_as(ctypes.c_void_p) for o in out],
                                B, T, Hq, Hkv, d, int(window), float(scale))
    _check(rc, "swa_bwd")
    return tuple(out)


def swa_lse(q_raw, k, alpha, beta, window: int, scale: float) -> np.ndarray:
    """Each base row's log-sum-exp of Eq. (4)'s scaled logits (natural log), fp64 [B,T,Hq]."""
    B, T, Hq, d = q_raw.shape
    Hkv = k.shape[2]
    q_raw, pq = _c(q_raw, np.uint16)
    k, pk = _c(k, np.uint16)
    alpha, pa = _c(alpha, np.float32)
    beta, pb = _c(beta, np.float32)
    out = np.zeros((B, T, Hq), np.float64)
    rc = _load().oracle_swa_lse(pq, pk, pa, pb, out.ctypes.data_as(ctypes.c_void_p), B, T, Hq, Hkv, d,
                                int(window), float(scale))
    _check(rc, "swa_lse")
    return out


def xattn_lse(qc_raw, pos, k, alpha_c, beta_c, scale: float) -> np.ndarray:
    """Each copy row's log-sum-exp of Eq. (5)'s scaled logits over keys 0..pos (natural log),
    fp64 [B,T_out,Hq]."""
    B, T_out, Hq, d = qc_raw.shape
    T_kv, Hkv = k.shape[1], k.shape[2]
    qc_raw, pq = _c(qc_raw, np.uint16)
    pos, pp = _c(pos, np.int32)
    k, pk = _c(k, np.uint16)
    alpha_c, pa = _c(alpha_c, np.float32)
    beta_c, pb = _c(beta_c, np.float32)
    out = np.zeros((B, T_out, Hq), np.float64)
    rc = _load().oracle_xattn_lse(pq, pp, pk, pa, pb, out.ctypes.data_as(ctypes.c_void_p), B, T_out, T_kv, Hq, Hkv,
                                  d, float(scale))
    _check(rc, "xattn_lse")
    return out


def xattn_bwd(qc_raw, pos, k, v, alpha_c, beta_c, dOc, scale: float):
    """Gradient of Eq. (5) with the copies' scale-offset for an output gradient dOc (bf16 bits
    [B,T_out,Hq,d]): returns fp64 (dqc_raw [B,T_out,Hq,d], dk, dv [B,T_kv,Hkv,d] -- the copies'
    share only --, dalpha_c, dbeta_c [Hq,d])."""
    B, T_out, Hq, d = qc_raw.shape
    T_kv, Hkv = k.shape[1], k.shape[2]
    assert k.shape == v.shape == (B, T_kv, Hkv, d) and dOc.shape == qc_raw.shape
    qc_raw, pq = _c(qc_raw, np.uint16)
    pos, pp = _c(pos, np.int32)
    k, pk = _c(k, np.uint16)
    v, pv = _c(v, np.uint16)
    alpha_c, pa = _c(alpha_c, np.float32)
    beta_c, pb = _c(beta_c, np.float32)
    dOc, pg = _c(dOc, np.uint16)
    out = [np.zeros(s, np.float64) for s in ((B, T_out, Hq, d), (B, T_kv, Hkv, d), (B, T_kv, Hkv, d),
                                             (Hq, d), (Hq, d))]
    rc = _load().oracle_xattn_bwd(pq, pp, pk, pv, pa, pb, pg, *[o.ctypes.data_as(ctypes.c_void_p) for o in out],
                                  B, T_out, T_kv, Hq, Hkv, d, float(scale))
    _check(rc, "xattn_bwd")
    return tuple(out)


def swa_rows(q_raw, k, v, alpha, beta, window: int, scale: float, b_idx, t_idx) -> np.ndarray:
    """Eq. (4) at the listed (b, t) rows only; returns fp64 [n, Hq, d]."""
    B, T, Hq, d = q_raw.shape
    Hkv = k.shape[2]
    q_raw, pq = _c(q_raw, np.uint16)
    k, pk = _c(k, np.uint16)
    v, pv = _c(v, np.uint16)
    alpha, pa = _c(alpha, np.float32)
    beta, pb = _c(beta, np.float32)
    bi, pbi = _c(b_idx, np.int32)
    ti, pti = _c(t_idx, np.int32)
    n = bi.size
    o = np.zeros((n, Hq, d), np.float64)
    rc = _load().oracle_swa_rows(pq, pk, pv, pa, pb, o.ctypes.data_as(ctypes.c_void_p),
                                 B, T, Hq, Hkv, d, int(window), float(scale), pbi, pti, n)
    _check(rc, "swa_rows")
    return o


def xattn(qc_raw, pos, k, v, alpha_c, beta_c, scale: float) -> np.ndarray:
    """Eq. (5) for copies at original positions pos [B,T_out] over base k/v [B,T_kv,Hkv,d]."""
    B, T_out, Hq, d = qc_raw.shape
    T_kv, Hkv = k.shape[1], k.shape[2]
    qc_raw, pq = _c(qc_raw, np.uint16)
    pos, pp = _c(pos, np.int32)
    k, pk = _c(k, np.uint16)
    v, pv = _c(v, np.uint16)
    alpha_c, pa = _c(alpha_c, np.float32)
    beta_c, pb = _c(beta_c, np.float32)
    oc = np.zeros((B, T_out, Hq, d), np.float64)
    rc = _load().oracle_xattn(pq, pp, pk, pv, pa, pb, oc.ctypes.data_as(ctypes.c_void_p),
                              B, T_out, T_kv, Hq, Hkv, d, float(scale))
    _check(rc, "xattn")
    return oc


def decode_step(q_new, qc_new, k_new, v_new, k_cache, v_cache, cache_len,
                alpha, beta, alpha_c, beta_c, window: int, scale: float):
    """One decode step.  Updates k_cache, v_cache (uint16 [B,L_max,Hkv,d]) and
    cache_len (int32 [B]) in place; returns (o, oc) fp64 [B, Hq, d]."""
    B, Hq, d = q_new.shape
    L_max, Hkv = k_cache.shape[1], k_cache.shape[2]
    for a, dt in ((k_cache, np.uint16), (v_cache, np.uint16), (cache_len, np.int32)):
        if not (a.flags.c_contiguous and a.dtype == dt):
            raise TypeError("cache arrays must be C-contiguous and of the documented dtype")
    q_new, p1 = _c(q_new, np.uint16)
    qc_new, p2 = _c(qc_new, np.uint16)
    k_new, p3 = _c(k_new, np.uint16)
    v_new, p4 = _c(v_new, np.uint16)
    arrs = [_c(x, np.float32) for x in (alpha, beta, alpha_c, beta_c)]
    o = np.zeros((B, Hq, d), np.float64)
    oc = np.zeros((B, Hq, d), np.float64)
    P = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    rc = _load().oracle_decode_step(p1, p2, p3, p4, P(k_cache), P(v_cache), P(cache_len), L_max,
                                    arrs[0][1], arrs[1][1], arrs[2][1], arrs[3][1], P(o), P(oc),
                                    B, Hq, Hkv, d, int(window), float(scale))
    _check(rc, "decode_step")
    return o, oc
