"""Seeded synthetic inputs for the Orthros per-layer attention operator.

This module only draws random numbers and lays them out; it holds none of the
operator's arithmetic.  Both the fp64 oracle (``oracle/``) and the CUDA path
(``long_context_attention_orthros_gb300``) are fed from here, so the two sides
see the same bytes.

Workloads follow the shapes of the pages' experiments (Orthros: Phase-Aware
Heterogeneous Attention, Sec. 4.5 prefill on 8B-class layers up to 1M tokens,
Sec. 4.6 batch-2 decode after a 128K prompt; Sec. 3.2 table of modes for the
copy layouts):

* bf16 tensors are returned as ``numpy.uint16`` bit patterns (round to nearest
  even from float32 draws), fp32 tensors as ``numpy.float32``.
* Q_raw / K / V / Q'_raw ~ N(0, 1); alpha, alpha' ~ 1 + N(0, 0.1);
  beta, beta' ~ N(0, 0.1).
* Layout is token-major ``[B, T, H, d]`` with d contiguous.

Every stream of random numbers is a Philox generator keyed by
``SeedSequence([seed, tensor_tag, chunk])``, so a tensor is reproducible chunk
by chunk and independent of how many threads produce it.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

# Tags that key the random streams of each tensor.
_TAGS = {
    "q_raw": 1, "k": 2, "v": 3, "qc_raw": 4, "alpha": 5, "beta": 6,
    "alpha_c": 7, "beta_c": 8, "pos": 9, "needle": 10,
    "q_new": 11, "qc_new": 12, "k_new": 13, "v_new": 14,
    "k_cache": 15, "v_cache": 16, "dO": 17, "dOc": 18,
}

_CHUNK = 1 << 22  # elements per independently keyed chunk


def _gen(seed: int, tag: str, chunk: int = 0) -> np.random.Generator:
    ss = np.random.SeedSequence([int(seed), _TAGS[tag], int(chunk)])
    return np.random.Generator(np.random.Philox(ss))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return the bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(seed: int, tag: str, shape, std: float = 1.0, threads: int | None = None) -> np.ndarray:
    """N(0, std^2) draws rounded to bf16, produced in independently keyed chunks."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.uint16)
    nchunks = max(1, math.ceil(n / _CHUNK))

    def fill(c: int) -> None:
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        x = _gen(seed, tag, c).standard_normal(hi - lo, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[lo:hi] = bf16_bits(x)

    if nchunks == 1:
        fill(0)
    else:
        workers = threads or min(16, os.cpu_count() or 1)
        with ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(fill, range(nchunks)))
    return out.reshape(shape)


def scale_offset(seed: int, Hq: int, d: int, prefix: str = "") -> tuple[np.ndarray, np.ndarray]:
    """alpha ~ 1 + N(0, 0.1), beta ~ N(0, 0.1), both fp32 [Hq, d]."""
    a = 1.0 + 0.1 * _gen(seed, "alpha" + prefix).standard_normal((Hq, d), dtype=np.float32)
    b = 0.1 * _gen(seed, "beta" + prefix).standard_normal((Hq, d), dtype=np.float32)
    return a.astype(np.float32), b.astype(np.float32)


@dataclass(frozen=True)
class PrefillConfig:
    """A prefill / SFT / PT-style layer: base SWA over T tokens plus T_out copies."""
    name: str
    B: int
    T: int
    Hq: int
    Hkv: int
    d: int
    window: int = 128
    T_out: int = 1
    # copies stored physically after the base tokens in one [B, T+T_out, Hq, d] buffer
    appended: bool = False
    # copy positions: "last" = the last T_out positions in order; "shuffled" = the
    # same set in a seeded random physical order
    positions: str = "last"
    needle_frac: float = 0.0   # fraction of key rows scaled by needle_scale
    needle_scale: float = 4.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


@dataclass(frozen=True)
class DecodeConfig:
    """A batch of sequences with a seeded KV cache, then `steps` decode steps."""
    name: str
    B: int
    T0: int
    steps: int
    Hq: int
    Hkv: int
    d: int
    window: int = 128
    fill_unused: int = 0x7FC0  # bf16 NaN in cache rows never written: any stray read shows

    @property
    def L_max(self) -> int:
        return self.T0 + self.steps

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# The five workloads: tiny prefill, 8B-class 128K prefill, batch-2 decode after a
# 128K prompt, SFT layer with an appended shuffled answer span, 1M-token prefill.
CONFIGS = {
    "tiny_prefill": PrefillConfig("tiny_prefill", B=1, T=512, Hq=2, Hkv=1, d=64),
    "prefill_128k": PrefillConfig("prefill_128k", B=2, T=131072, Hq=32, Hkv=8, d=128),
    "decode_128k": DecodeConfig("decode_128k", B=2, T0=131072, steps=128, Hq=32, Hkv=8, d=128),
    # the same layer and cache length at batch 8 (decode's batch dependence)
    "decode_128k_b8": DecodeConfig("decode_128k_b8", B=8, T0=131072, steps=32, Hq=32, Hkv=8, d=128),
    "sft_16k": PrefillConfig("sft_16k", B=4, T=16384, Hq=32, Hkv=8, d=128, T_out=2048,
                             appended=True, positions="shuffled"),
    "prefill_1m": PrefillConfig("prefill_1m", B=1, T=1048576, Hq=32, Hkv=8, d=128,
                                needle_frac=0.001),
    # a profiling-sized prefill with the same layer shape (inputs still larger than L2)
    "prefill_16k": PrefillConfig("prefill_16k", B=1, T=16384, Hq=32, Hkv=8, d=128),
    # one sequence of the SFT layer (profiling size)
    "sft_16k_1": PrefillConfig("sft_16k_1", B=1, T=16384, Hq=32, Hkv=8, d=128, T_out=2048,
                               appended=True, positions="shuffled"),
}

SEEDS = {"tiny_prefill": 1, "prefill_128k": 2, "decode_128k": 3, "sft_16k": 4, "prefill_1m": 5,
         "prefill_16k": 6, "sft_16k_1": 7, "decode_128k_b8": 8}


@dataclass
class PrefillInputs:
    cfg: PrefillConfig
    q_raw: np.ndarray     # bf16 bits; [B, T, Hq, d], or [B, T+T_out, Hq, d] when appended
    k: np.ndarray         # bf16 bits [B, T, Hkv, d]
    v: np.ndarray         # bf16 bits [B, T, Hkv, d]
    qc_raw: np.ndarray    # bf16 bits [B, T_out, Hq, d] (a view of q_raw's tail when appended)
    pos: np.ndarray       # int32 [B, T_out] original positions of the copies
    alpha: np.ndarray     # fp32 [Hq, d]
    beta: np.ndarray
    alpha_c: np.ndarray
    beta_c: np.ndarray
    needles: np.ndarray = field(default_factory=lambda: np.zeros((0,), np.int64))

    @property
    def q_base(self) -> np.ndarray:
        """The base-stream rows of q_raw ([B, T, Hq, d] view)."""
        return self.q_raw[:, : self.cfg.T]


def make_prefill(cfg: PrefillConfig, seed: int) -> PrefillInputs:
    B, T, Hq, Hkv, d, T_out = cfg.B, cfg.T, cfg.Hq, cfg.Hkv, cfg.d, cfg.T_out
    rows = T + T_out if cfg.appended else T
    if cfg.appended:
        q_all = np.empty((B, rows, Hq, d), dtype=np.uint16)
        q_all[:, :T] = normal_bf16(seed, "q_raw", (B, T, Hq, d))
        q_all[:, T:] = normal_bf16(seed, "qc_raw", (B, T_out, Hq, d))
        q_raw, qc_raw = q_all, q_all[:, T:]
    else:
        q_raw = normal_bf16(seed, "q_raw", (B, T, Hq, d))
        qc_raw = normal_bf16(seed, "qc_raw", (B, T_out, Hq, d))
    k = normal_bf16(seed, "k", (B, T, Hkv, d))
    v = normal_bf16(seed, "v", (B, T, Hkv, d))
    needles = np.zeros((0,), np.int64)
    if cfg.needle_frac > 0:
        n = max(1, round(cfg.needle_frac * T))
        g = _gen(seed, "needle")
        needles = np.sort(g.choice(T, size=n, replace=False))
        kf = bf16_to_f32(k[:, needles]) * np.float32(cfg.needle_scale)  # power of two: exact
        k[:, needles] = bf16_bits(kf)
    base_pos = np.arange(T - T_out, T, dtype=np.int32)
    if cfg.positions == "shuffled":
        g = _gen(seed, "pos")
        pos = np.stack([g.permutation(base_pos) for _ in range(B)]).astype(np.int32)
    else:
        pos = np.tile(base_pos, (B, 1)).astype(np.int32)
    alpha, beta = scale_offset(seed, Hq, d)
    alpha_c, beta_c = scale_offset(seed, Hq, d, prefix="_c")
    return PrefillInputs(cfg, q_raw, k, v, qc_raw, pos, alpha, beta, alpha_c, beta_c, needles)


@dataclass
class DecodeInputs:
    cfg: DecodeConfig
    k_cache: np.ndarray   # bf16 bits [B, L_max, Hkv, d]; rows >= T0 hold cfg.fill_unused
    v_cache: np.ndarray
    cache_len: np.ndarray  # int32 [B], all T0
    q_new: np.ndarray     # bf16 bits [steps, B, Hq, d]
    qc_new: np.ndarray
    k_new: np.ndarray     # bf16 bits [steps, B, Hkv, d]
    v_new: np.ndarray
    alpha: np.ndarray
    beta: np.ndarray
    alpha_c: np.ndarray
    beta_c: np.ndarray


def make_decode(cfg: DecodeConfig, seed: int) -> DecodeInputs:
    B, T0, S, Hq, Hkv, d = cfg.B, cfg.T0, cfg.steps, cfg.Hq, cfg.Hkv, cfg.d
    k_cache = np.full((B, cfg.L_max, Hkv, d), cfg.fill_unused, dtype=np.uint16)
    v_cache = np.full((B, cfg.L_max, Hkv, d), cfg.fill_unused, dtype=np.uint16)
    k_cache[:, :T0] = normal_bf16(seed, "k_cache", (B, T0, Hkv, d))
    v_cache[:, :T0] = normal_bf16(seed, "v_cache", (B, T0, Hkv, d))
    alpha, beta = scale_offset(seed, Hq, d)
    alpha_c, beta_c = scale_offset(seed, Hq, d, prefix="_c")
    return DecodeInputs(
        cfg, k_cache, v_cache, np.full((B,), T0, dtype=np.int32),
        normal_bf16(seed, "q_new", (S, B, Hq, d)), normal_bf16(seed, "qc_new", (S, B, Hq, d)),
        normal_bf16(seed, "k_new", (S, B, Hkv, d)), normal_bf16(seed, "v_new", (S, B, Hkv, d)),
        alpha, beta, alpha_c, beta_c)


def reduced(cfg, **kw):
    """A copy of a config with some sizes changed (for parity cases the oracle finishes fast)."""
    from dataclasses import replace
    return replace(cfg, **kw)
