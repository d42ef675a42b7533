"""Benchmark of the Orthros per-layer attention operator on GB300.

Default workload: 8B-class prefill, batch 2 x 131072 tokens, 32 query heads /
8 KV heads, d=128, w=128, one output copy per sequence at its last position.
One step = base SWA (Eq. 4) over every token + the copies' cross-attention
(Eq. 5), i.e. the whole prefill hot path.  The same JSON line carries further
legs, each with its own roofline object:

* ``decode``      batch 2, 131072-token cache, 128 consecutive fused decode steps
                  (eager and replayed as one CUDA graph)
* ``decode_b8``   the same at batch 8 (32 steps)
* ``gradient``    both streams' attention gradient on the prefill inputs
* ``sft``         the SFT layer: batch 4 x 16384 tokens + 2048 appended copies each
* ``prefill_1m``  one 1048576-token sequence with scaled key rows

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl orthros|reference]
                    [--legs prefill,e2e,decode,decode_b8,gradient,sft,prefill_1m,cpu]

Under torchrun each rank runs the same workload on its own GPU (independent
sequences, weak scaling, no data-path collective); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from synthetic import CONFIGS, SEEDS, make_decode, make_prefill, reduced  # noqa: E402

METRIC = "prefill tokens/s (SWA+1 global query) at 128K; decode steps/s; % of HBM peak"
KERNEL_SRC = os.path.join(ROOT, "long_context_attention_orthros_gb300", "csrc")
ALL_LEGS = ("prefill", "e2e", "decode", "decode_b8", "gradient", "sft", "prefill_1m", "cpu")
# the nominal HBM3e bandwidth of a GB300 (the ~8 TB/s figure the target is stated against)
HBM_NAMEPLATE_GBS = 8000.0
SWA_SOURCES = ("swa_fwd.cu", "swa_tc.cu", "tc.cuh", "common.cuh", "kernels.cuh")
DECODE_SOURCES = ("decode_step.cu", "xattn.cuh", "common.cuh", "kernels.cuh")
BWD_SOURCES = ("attn_bwd.cuh", "attn_bwd.cu", "attn_bwd_d128.cu", "tc.cuh", "common.cuh", "kernels.cuh")
XTC_SOURCES = ("xattn_tc.cu", "tc.cuh", "common.cuh", "kernels.cuh")
XATTN_SOURCES = ("xattn_fwd.cu", "xattn.cuh", "common.cuh", "kernels.cuh")
L2_NOTE = "inputs larger than L2 (129 MB), no flush"


# ----------------------------------------------------------------- helpers

def _peaks():
    """Roofline denominators: the measured copy bandwidth and cuBLAS bf16 rates of this machine's
    GB300s (burst, and sustained under the power cap), else the recipe's fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm": float(d["hbm_gbs"]), "bf16": float(d["bf16_tflops"]),
                "bf16_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "kind": "measured"}
    return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "kind": "fallback"}


def kernel_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(KERNEL_SRC, n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profile_traffic(name, sources):
    """DRAM bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum) from a committed
    summary under profiles/, if it was taken on the kernel sources as they are now; else None."""
    path = os.path.join(ROOT, "profiles", f"{name}.json")
    if not os.path.exists(path):
        return None, None
    with open(path) as f:
        d = json.load(f)
    if d.get("kernel_source_sha256_16") != kernel_hash(*sources):
        return None, None
    return d.get("dram_bytes_per_launch"), f"profiles/{name}.json"


def step_roofline(swa_nbytes, step_nbytes, ms, peaks, name):
    """The prefill step as one unit: with few copies its two kernels run at once (the copies'
    split-KV pass on the SMs the SWA kernel leaves), so the step's algorithmic bytes over its
    time.  traffic: the two kernels' one-pass DRAM captures, when both are current."""
    gbs = step_nbytes / (ms / 1e3) / 1e9
    t_swa, s_swa = profile_traffic(f"swa_fwd_{name}", SWA_SOURCES)
    t_x, s_x = profile_traffic(f"xattn_fwd_{name}", XATTN_SOURCES)
    both = t_swa is not None and t_x is not None
    return {"kernel": "prefill step: swa_tc_kernel with the copies' split-KV pass beside it", "bound": "hbm",
            "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s", "frac": gbs / peaks["hbm"],
            "frac_nameplate": gbs / HBM_NAMEPLATE_GBS, "nameplate_peak": HBM_NAMEPLATE_GBS,
            "traffic": t_swa + t_x if both else None, "traffic_source": f"{s_swa} + {s_x}" if both else None,
            "peak_kind": peaks["kind"], "algorithmic_bytes": step_nbytes, "swa_algorithmic_bytes": swa_nbytes,
            "ms_per_launch": ms, "concurrent": True}


def hbm_roofline(kernel, nbytes, ms, peaks, traffic_name=None, sources=()):
    gbs = nbytes / (ms / 1e3) / 1e9
    traffic, src = profile_traffic(traffic_name, sources) if traffic_name else (None, None)
    return {"kernel": kernel, "bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
            "frac": gbs / peaks["hbm"], "frac_nameplate": gbs / HBM_NAMEPLATE_GBS,
            "nameplate_peak": HBM_NAMEPLATE_GBS, "traffic": traffic, "traffic_source": src,
            "peak_kind": peaks["kind"], "algorithmic_bytes": nbytes, "ms_per_launch": ms}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        busy = [s for s in sm if s > 0]
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def allreduce_max(x: float, world: int) -> float:
    """Max of a float over all ranks (timing only; no data-path collective)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def swa_bytes(B, T, Hq, Hkv, d) -> int:
    """Algorithmic bytes of Eq. (4) over B x T tokens: Q and O (Hq heads), K and V, once each."""
    return B * T * (2 * Hq + 2 * Hkv) * d * 2


def swa_pairs(B, T, Hq, w) -> int:
    """(query row, key) pairs of Eq. (4): row t sees min(t + 1, w) keys."""
    n = min(T, w)
    return B * Hq * (n * (n + 1) // 2 + (T - n) * w)


def xattn_bytes(pos, Hq, Hkv, d, T_kv) -> int:
    """Algorithmic bytes of Eq. (5): each sequence's K/V rows 0..max(pos) once, Q' and O' once."""
    B, T_out = pos.shape
    kv = sum(min(int(pos[b].max()) + 1, T_kv) for b in range(B)) * Hkv * d * 2 * 2 if T_out else 0
    return kv + B * T_out * Hq * d * 2 * 2


def launches_per_prefill_step(cfg) -> int:
    """Kernels one prefill step launches: SWA, the copies' kernel, and the combine kernel when
    the split-KV plan gives a row more than one partial (mirror of xattn_fwd.cu's plan)."""
    G = cfg.Hq // cfg.Hkv
    if cfg.T_out * G >= 256:
        return 2  # tensor-memory copies kernel, no partials
    rows = cfg.T_out * G
    wk = 4 if rows <= 16 else 1
    row_tiles = math.ceil(rows / (16 * (4 // wk)))
    base = cfg.B * cfg.Hkv * row_tiles
    splits = min(max(1, math.ceil(304 / base)), math.ceil(cfg.T / 256))
    chunk = math.ceil(math.ceil(cfg.T / splits) / 64) * 64
    splits = math.ceil(cfg.T / chunk)
    n_part = splits if rows <= 8 else splits * wk  # at most 8 rows: one partial per CTA
    return 2 + (0 if n_part == 1 else 1)


def bwd_launches_per_call(T_out, G, window) -> int:
    """Kernels one orthros_attn_bwd call launches with both forwards' log-sum-exp given (mirror of
    attn_bwd.cuh): fp16 K; the base stream's rows pass (fp16 q and D) and dq (the key-band kernel
    sums dalpha / dbeta in its epilogue for G = 4, 8 when the band fits five 32-key slots, else a
    separate pass sums them); the copies' rows pass and dq; one dk/dv launch for both streams."""
    units = 128 // G if G >= 4 else 0
    band = units > 0 and max(((1 << 20) + a + units - 1) // 32 - ((1 << 20) + a - window + 1) // 32 + 1
                             for a in range(0, 32, units)) <= 5
    base = 2 if band and G <= 8 else 3
    return 1 + base + (2 if T_out > 0 else 0) + 1


def _events(n):
    import torch
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def _mean_ms(pairs):
    return statistics.mean(a.elapsed_time(b) for a, b in pairs)


# ----------------------------------------------------------------- CPU oracle baselines

def oracle_prefill_rate(inp, target_s: float = 8.0, threads: int | None = None):
    """The fp64 oracle on a bounded sample of a prefill workload: n base rows in the middle of
    each sequence (all heads), sized to about target_s, plus the copies' whole cross-attention.
    Returns (extrapolated tokens/s of the full step, threads, sample description, wall s)."""
    import oracle
    cfg = inp.cfg
    if threads is not None:
        oracle.set_num_threads(threads)
    try:
        q = inp.q_base
        t_x0 = time.perf_counter()
        oracle.xattn(np.ascontiguousarray(inp.qc_raw), inp.pos, inp.k, inp.v, inp.alpha_c, inp.beta_c, cfg.scale)
        t_x = time.perf_counter() - t_x0
        n = 64
        while True:
            mid = cfg.T // 2
            t_idx = (mid + np.arange(n) // cfg.B) % cfg.T
            b_idx = np.arange(n) % cfg.B
            t0 = time.perf_counter()
            oracle.swa_rows(q, inp.k, inp.v, inp.alpha, inp.beta, cfg.window, cfg.scale, b_idx, t_idx)
            dt = time.perf_counter() - t0
            if dt >= target_s / 2 or n >= cfg.B * cfg.T:
                break
            n = min(cfg.B * cfg.T, n * 4 if dt < target_s / 16 else n * 2)
        nthreads = oracle.num_threads()
    finally:
        if threads is not None:
            oracle.set_num_threads(os.cpu_count() or 1)
    per_token = dt / n + t_x / (cfg.B * cfg.T)
    sample = (f"{n} of {cfg.B * cfg.T} base tokens x {cfg.Hq} heads (fp64 SWA rows, {dt:.2f} s) + "
              f"{cfg.B * cfg.T_out} copies over {cfg.T} keys ({t_x:.2f} s); rate extrapolated to the full step")
    return 1.0 / per_token, nthreads, sample, dt + t_x


def oracle_decode_rate(steps: int = 3):
    """The fp64 oracle's decode step on the batch-2, 131072-token cache (all threads): the
    first `steps` of the 128 steps, each appending and attending over the whole cache."""
    import oracle
    cfg = CONFIGS["decode_128k"]
    inp = make_decode(cfg, SEEDS[cfg.name])
    kc, vc, cl = inp.k_cache, inp.v_cache, inp.cache_len.copy()
    t0 = time.perf_counter()
    for i in range(steps):
        oracle.decode_step(inp.q_new[i], inp.qc_new[i], inp.k_new[i], inp.v_new[i], kc, vc, cl, inp.alpha, inp.beta,
                           inp.alpha_c, inp.beta_c, cfg.window, cfg.scale)
    dt = time.perf_counter() - t0
    return {"value": steps / dt, "unit": "steps/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"the first {steps} of the {cfg.steps} steps of {cfg.name} (B={cfg.B}, cache {cfg.T0}); "
                      f"{dt:.2f} s wall"}


def cpu_baselines(inp):
    prefill_rate, threads, sample, _ = oracle_prefill_rate(inp)
    one_rate, _, one_sample, _ = oracle_prefill_rate(inp, target_s=2.0, threads=1)
    return {"value": prefill_rate, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample,
            "single_thread": {"value": one_rate, "unit": "tokens/s", "cores": 1, "sample": one_sample},
            "decode": oracle_decode_rate()}


def _config_line(cfg):
    return {"workload": cfg.name, "B": cfg.B, "T": cfg.T, "Hq": cfg.Hq, "Hkv": cfg.Hkv, "d": cfg.d,
            "window": cfg.window, "T_out": cfg.T_out, "l2": L2_NOTE}


def run_reference(args):
    """The reference arm: the fp64 oracle as it stands on the host cores.  Each step is a bounded
    sample of the prefill workload (a slice of the base rows, all heads, plus the copies'
    whole cross-attention); `value` is the rate extrapolated to the full step."""
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    cfg = _config(args)
    inp = make_prefill(cfg, SEEDS[cfg.name])
    import oracle
    oracle.build()
    rates, walls, descs, threads = [], [], "", 0
    for i in range(args.warmup + args.steps):
        r, threads, descs, wall = oracle_prefill_rate(inp, target_s=2.0)
        if i >= args.warmup:
            rates.append(r)
            walls.append(wall)
    value = statistics.mean(rates)
    ms = statistics.mean(walls) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "extrapolated": True,
        "full_step_ms_extrapolated": cfg.B * cfg.T / value * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _config_line(cfg),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": descs},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- GPU legs

def _upload_prefill(inp, dev):
    import torch

    def bf(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(dev)

    def f(x):
        return torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    cfg = inp.cfg
    q = bf(inp.q_raw)
    qc = q[:, cfg.T:] if cfg.appended else bf(inp.qc_raw)
    return {"q": q, "k": bf(inp.k), "v": bf(inp.v), "qc": qc, "pos": f(inp.pos), "a": f(inp.alpha),
            "b": f(inp.beta), "ac": f(inp.alpha_c), "bc": f(inp.beta_c)}


def time_prefill(g, cfg, dev, steps, warmup, world):
    """Time `steps` prefill steps after `warmup` untimed ones: one orthros_prefill_fwd call per
    step (for few copies it runs their split-KV pass on a second stream beside the SWA kernel),
    with CUDA events around the whole region on the launching stream.  Then each kernel alone
    (SWA on every SM, then the copies' pass), with events around each call, for the per-kernel
    rooflines."""
    import torch
    import long_context_attention_orthros_gb300 as orth
    B, T, Hq, d, T_out = cfg.B, cfg.T, cfg.Hq, cfg.d, cfg.T_out
    o = torch.empty((B, T, Hq, d), dtype=torch.bfloat16, device=dev)
    oc = torch.empty((B, T_out, Hq, d), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(orth.prefill_workspace_size(B, T, T_out, Hq, cfg.Hkv, d), 256), dtype=torch.uint8,
                     device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        orth.prefill_fwd(g["q"], g["k"], g["v"], g["a"], g["b"], g["qc"], g["pos"], g["ac"], g["bc"],
                         window=cfg.window, scale=cfg.scale, out=o, out_c=oc, workspace=ws, dev_err=err)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    _barrier(world)
    torch.cuda.synchronize()
    t0, t1 = _events(2)
    t0.record(stream)
    for _ in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    _barrier(world)
    ms = allreduce_max(t0.elapsed_time(t1) / steps, world)
    ev_s, ev_x = [], []
    for _ in range(max(3, min(steps, 10))):
        e = _events(3)
        e[0].record(stream)
        orth.swa_fwd(g["q"], g["k"], g["v"], g["a"], g["b"], window=cfg.window, scale=cfg.scale, out=o, dev_err=err)
        e[1].record(stream)
        orth.xattn_fwd(g["qc"], g["pos"], g["k"], g["v"], g["ac"], g["bc"], scale=cfg.scale, out=oc, workspace=ws,
                       dev_err=err)
        e[2].record(stream)
        ev_s.append((e[0], e[1]))
        ev_x.append((e[1], e[2]))
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error word {int(err.item())}"
    return ms, _mean_ms(ev_s), _mean_ms(ev_x), o, oc, ws, err


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def run_e2e(g, o, oc, ws, err, inp, cfg, dev, steps, world):
    """End to end through the public API: pinned host inputs uploaded, the step computed and its
    outputs downloaded inside the timed region, every step.  Pipelined by 8K-row chunks on
    three streams: the upload of chunk c+1, the SWA of chunk c (orthros_swa_fwd_rows; its key
    halo is in chunk c-1) and the download of chunk c-1 overlap; the copies' cross-attention
    runs once the last K/V chunk is on the device."""
    import torch
    import long_context_attention_orthros_gb300 as orth
    B, T, Hq, d, T_out = cfg.B, cfg.T, cfg.Hq, cfg.d, cfg.T_out

    def pinned(x, dtype):
        t = torch.empty(x.shape, dtype=dtype, pin_memory=True)
        t.numpy()[...] = x.view(np.int16) if dtype == torch.int16 else x
        return t

    h = {"q": pinned(inp.q_raw, torch.int16), "k": pinned(inp.k, torch.int16), "v": pinned(inp.v, torch.int16),
         "qc": pinned(np.ascontiguousarray(inp.qc_raw), torch.int16), "pos": pinned(inp.pos, torch.int32),
         "a": pinned(inp.alpha, torch.float32), "b": pinned(inp.beta, torch.float32),
         "ac": pinned(inp.alpha_c, torch.float32), "bc": pinned(inp.beta_c, torch.float32)}
    ho = torch.empty((B, T, Hq, d), dtype=torch.int16, pin_memory=True)
    hoc = torch.empty((B, T_out, Hq, d), dtype=torch.int16, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in h.values())
    d2h = ho.numel() * 2 + hoc.numel() * 2
    stream = torch.cuda.current_stream(dev)
    chunk = 8192
    cuts = list(range(0, T, chunk)) + [T]
    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))

    def up(key, r0=None, r1=None):
        dst = g[key].view(torch.int16) if key in ("q", "k", "v", "qc") else g[key]
        if r0 is None:
            dst.copy_(h[key], non_blocking=True)
        else:
            for bb in range(B):
                dst[bb, r0:r1].copy_(h[key][bb, r0:r1], non_blocking=True)

    def e2e_step():
        start = torch.cuda.Event()
        start.record(stream)
        for st_ in (s_in, s_comp, s_out):
            st_.wait_event(start)
        with torch.cuda.stream(s_in):
            for key in ("a", "b", "ac", "bc", "qc", "pos"):
                up(key)
        for c0, c1 in zip(cuts[:-1], cuts[1:]):
            with torch.cuda.stream(s_in):
                for key in ("q", "k", "v"):
                    up(key, c0, c1)
                landed = torch.cuda.Event()
                landed.record(s_in)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(landed)
                orth.swa_fwd_rows(g["q"], g["k"], g["v"], g["a"], g["b"], c0, c1, window=cfg.window,
                                  scale=cfg.scale, out=o, dev_err=err)
                done = torch.cuda.Event()
                done.record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done)
                for bb in range(B):
                    ho[bb, c0:c1].copy_(o.view(torch.int16)[bb, c0:c1], non_blocking=True)
        with torch.cuda.stream(s_comp):
            orth.xattn_fwd(g["qc"], g["pos"], g["k"], g["v"], g["ac"], g["bc"], scale=cfg.scale, out=oc,
                           workspace=ws, dev_err=err)
            done = torch.cuda.Event()
            done.record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(done)
            hoc.copy_(oc.view(torch.int16), non_blocking=True)
        for st_ in (s_in, s_comp, s_out):
            stream.wait_stream(st_)

    n = max(3, min(steps, 10))
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    _barrier(world)
    a0, a1 = _events(2)
    a0.record(stream)
    for _ in range(n):
        e2e_step()
    a1.record(stream)
    torch.cuda.synchronize()
    _barrier(world)
    ms = allreduce_max(a0.elapsed_time(a1) / n, world)
    assert int(err.item()) == 0
    return {"value": B * T * world / (ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": n}


def run_gradient(dev, world, g, o, oc, cfg, peaks, calls: int = 5):
    """The layer's attention gradient on the prefill inputs with seeded N(0, 1) output
    gradients: orthros_attn_bwd, both streams in one call, each with its forward's
    log-sum-exp (computed untimed beforehand)."""
    import torch
    import long_context_attention_orthros_gb300 as orth
    B, T, Hq, Hkv, d, T_out = cfg.B, cfg.T, cfg.Hq, cfg.Hkv, cfg.d, cfg.T_out
    gen = torch.Generator(device=dev)
    gen.manual_seed(SEEDS[cfg.name] + 17)
    dO = torch.randn((B, T, Hq, d), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
    dOc = torch.randn((B, T_out, Hq, d), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
    ws = torch.empty(orth.attn_bwd_workspace_size(B, T, T_out, Hq, Hkv, d), dtype=torch.uint8, device=dev)
    qc = g["qc"].contiguous()
    q = g["q"] if g["q"].shape[1] == T else g["q"][:, :T].contiguous()
    stream = torch.cuda.current_stream(dev)
    _, lse = orth.swa_fwd_lse(q, g["k"], g["v"], g["a"], g["b"], window=cfg.window, scale=cfg.scale)
    lsec = None
    if T_out > 0:
        _, lsec = orth.xattn_fwd(qc, g["pos"], g["k"], g["v"], g["ac"], g["bc"], scale=cfg.scale, lse=True)

    def call():
        return orth.attn_bwd(q, g["k"], g["v"], g["a"], g["b"], o, dO, qc, g["pos"], g["ac"], g["bc"], oc, dOc,
                             window=cfg.window, scale=cfg.scale, lse=lse, lsec=lsec, workspace=ws)

    for _ in range(3):
        grads = call()
    torch.cuda.synchronize()
    e0, e1 = _events(2)
    e0.record(stream)
    for _ in range(calls):
        grads = call()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = allreduce_max(e0.elapsed_time(e1) / calls, world)
    assert all(bool(torch.isfinite(t).all()) for t in grads)
    del grads, dO, dOc, ws, lse, lsec, q
    per_call = bwd_launches_per_call(T_out, Hq // Hkv, cfg.window)
    # algorithmic bytes: q_raw, o, dO (bf16) and each row's log-sum-exp read, K and V read, fp32
    # dq, dk, dv written, once each (both streams); dalpha / dbeta are [Hq, d]
    rows = B * (T + T_out) * Hq
    nbytes = 3 * rows * d * 2 + rows * 4 + 2 * B * T * Hkv * d * 2 + rows * d * 4 + 2 * B * T * Hkv * d * 4
    pos = g["pos"].cpu().numpy().astype(np.int64)
    pairs = swa_pairs(B, T, Hq, cfg.window) + Hq * int((pos + 1).sum())
    flops = 10 * d * pairs  # S, dP, dV, dK, dQ: 2 d flops each per (row, key) pair
    t_hbm = nbytes / (peaks["hbm"] * 1e9) * 1e3
    t_tc = flops / (peaks["bf16"] * 1e12) * 1e3
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    gbs = nbytes / (ms / 1e3) / 1e9
    tfs = flops / (ms / 1e3) / 1e12
    traffic, tsrc = profile_traffic(f"attn_bwd_{cfg.name}", BWD_SOURCES)
    roof = {"kernel": f"attn_bwd ({per_call} launches)", "bound": bound,
            "achieved": gbs if bound == "hbm" else tfs, "peak": peaks["hbm"] if bound == "hbm" else peaks["bf16"],
            "unit": "GB/s" if bound == "hbm" else "TFLOP/s", "frac": max(t_hbm, t_tc) / ms,
            "traffic": traffic, "traffic_source": tsrc, "peak_kind": peaks["kind"], "algorithmic_bytes": nbytes,
            "algorithmic_flops": flops,
            "roofline_ms": max(t_hbm, t_tc), "hbm_ms": t_hbm, "tensor_ms": t_tc, "tflops": tfs}
    return {"value": B * T * world / (ms / 1e3), "unit": "tokens/s", "ms_per_call": ms,
            "what": "attn_bwd: both streams' gradient in one call (dK/dV written once), each stream with its "
                    "forward's log-sum-exp", "roofline": roof, "gpu_launches": per_call * calls}


def run_decode(dev, world, peaks, name, reps: int = 3):
    """`steps` consecutive fused decode steps on a seeded 131072-token cache, eager and as one
    replayed CUDA graph; the cache length is reset between repetitions."""
    import torch
    import long_context_attention_orthros_gb300 as orth
    cfg = CONFIGS[name]
    inp = make_decode(cfg, SEEDS[cfg.name])
    B, Hq, Hkv, d, S = cfg.B, cfg.Hq, cfg.Hkv, cfg.d, cfg.steps

    def bf(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(dev)

    kc, vc = bf(inp.k_cache), bf(inp.v_cache)
    del inp.k_cache, inp.v_cache
    cl0 = torch.from_numpy(inp.cache_len).to(dev)
    cl = cl0.clone()
    qn, qcn, kn, vn = bf(inp.q_new), bf(inp.qc_new), bf(inp.k_new), bf(inp.v_new)
    a, b_, ac, bc = (torch.from_numpy(x).to(dev) for x in (inp.alpha, inp.beta, inp.alpha_c, inp.beta_c))
    ws = orth._binding.decode_workspace(B, cfg.L_max, Hq, Hkv, d, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    o = torch.empty((B, Hq, d), dtype=torch.bfloat16, device=dev)
    oc = torch.empty_like(o)
    stream = torch.cuda.current_stream(dev)

    def run_all():
        for i in range(S):
            orth.decode_step(qn[i], qcn[i], kn[i], vn[i], kc, vc, cl, a, b_, ac, bc, window=cfg.window,
                             scale=cfg.scale, o=o, oc=oc, workspace=ws, dev_err=err)

    def timed(fn):
        total = 0.0
        for _ in range(reps):
            cl.copy_(cl0)
            torch.cuda.synchronize()
            e0, e1 = _events(2)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            total += e0.elapsed_time(e1)
        return allreduce_max(total / (reps * S), world)

    cl.copy_(cl0)
    run_all()  # warm-up pass
    ms_step = timed(run_all)
    assert int(err.item()) == 0, f"decode device error {int(err.item())}"
    graph = torch.cuda.CUDAGraph()
    cl.copy_(cl0)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        run_all()
    gms_step = timed(graph.replay)
    assert int(err.item()) == 0, f"decode device error {int(err.item())} (graph)"
    avg_len = cfg.T0 + (S + 1) / 2
    step_bytes = int(B * avg_len * Hkv * d * 2 * 2)  # the whole cache's K and V, once per step
    roof = hbm_roofline("decode_step", step_bytes, ms_step, peaks, f"decode_step_{cfg.name}", DECODE_SOURCES)
    return {"value": world / (ms_step / 1e3), "unit": "steps/s", "ms_per_step": ms_step,
            "config": {"workload": cfg.name, "B": B, "cache_len": cfg.T0, "steps": S, "Hq": Hq, "Hkv": Hkv,
                       "d": d, "window": cfg.window},
            "roofline": roof,
            "cuda_graph": {"value": world / (gms_step / 1e3), "unit": "steps/s", "ms_per_step": gms_step,
                           "frac": step_bytes / (gms_step / 1e3) / 1e9 / peaks["hbm"],
                           "note": f"the {S} steps captured once and replayed"},
            "gpu_launches": 2 * reps * S}


def run_sft(dev, world, peaks, steps, warmup):
    """The SFT layer: base SWA over B x 16384 tokens and Eq. (5) for the 2048 answer copies of
    each sequence, stored after the base tokens with shuffled original positions."""
    cfg = CONFIGS["sft_16k"]
    inp = make_prefill(cfg, SEEDS[cfg.name])
    g = _upload_prefill(inp, dev)
    ms, swa_ms, x_ms, *_ = time_prefill(g, cfg, dev, steps, warmup, world)
    B, T, Hq, Hkv, d = cfg.B, cfg.T, cfg.Hq, cfg.Hkv, cfg.d
    pos = inp.pos.astype(np.int64)
    flops = 4 * d * Hq * int((pos + 1).sum())
    xb = xattn_bytes(inp.pos, Hq, Hkv, d, T)
    tfs = flops / (x_ms / 1e3) / 1e12
    t_tc = flops / (peaks["bf16_sustained"] * 1e12) * 1e3
    t_hbm = xb / (peaks["hbm"] * 1e9) * 1e3
    traffic, tsrc = profile_traffic(f"xattn_tc_{cfg.name}", XTC_SOURCES)
    return {"value": B * T * world / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
            "copies_per_s": B * cfg.T_out * world / (ms / 1e3), "config": _config_line(cfg),
            "roofline": {"kernel": "xattn_tc", "bound": "tensor" if t_tc >= t_hbm else "hbm", "achieved": tfs,
                         "peak": peaks["bf16_sustained"], "unit": "TFLOP/s", "frac": max(t_tc, t_hbm) / x_ms,
                         "frac_of_burst": tfs / peaks["bf16"], "traffic": traffic, "traffic_source": tsrc,
                         "peak_kind": peaks["kind"] + " sustained",
                         "algorithmic_flops": flops, "algorithmic_bytes": xb, "ms_per_launch": x_ms},
            "swa": hbm_roofline("swa_tc", swa_bytes(B, T, Hq, Hkv, d), swa_ms, peaks, f"swa_fwd_{cfg.name}",
                                SWA_SOURCES),
            "gpu_launches": steps * launches_per_prefill_step(cfg)}


def run_prefill_1m(dev, world, peaks, steps, warmup):
    """One 1048576-token sequence (0.1% of key rows scaled x4) with its copy at the last position."""
    cfg = CONFIGS["prefill_1m"]
    inp = make_prefill(cfg, SEEDS[cfg.name])
    g = _upload_prefill(inp, dev)
    pos = inp.pos
    del inp
    ms, swa_ms, x_ms, *_ = time_prefill(g, cfg, dev, steps, warmup, world)
    B, T, Hq, Hkv, d = cfg.B, cfg.T, cfg.Hq, cfg.Hkv, cfg.d
    nbytes = swa_bytes(B, T, Hq, Hkv, d)
    step_bytes = nbytes + xattn_bytes(pos, Hq, Hkv, d, T)
    return {"value": B * T * world / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms, "steps": steps,
            "config": _config_line(cfg), "xattn_alone_ms": x_ms,
            "roofline": step_roofline(nbytes, step_bytes, ms, peaks, cfg.name),
            "swa_alone": hbm_roofline("swa_tc", nbytes, swa_ms, peaks, f"swa_fwd_{cfg.name}", SWA_SOURCES),
            "gpu_launches": steps * launches_per_prefill_step(cfg)}


def _config(args):
    cfg = CONFIGS[args.config]
    return reduced(cfg, B=args.batch) if args.batch else cfg


def run_gpu(args):
    import torch

    legs = set(args.legs.split(",")) if args.legs else set(ALL_LEGS)
    unknown = legs - set(ALL_LEGS)
    if unknown:
        raise SystemExit(f"unknown legs: {sorted(unknown)}")
    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    import long_context_attention_orthros_gb300  # noqa: F401  (fails loudly without the library)
    peaks = _peaks()
    warmup = max(3, args.warmup)

    cfg = _config(args)
    inp = make_prefill(cfg, SEEDS[cfg.name] + 1000 * rank)
    B, T, Hq, Hkv, d = cfg.B, cfg.T, cfg.Hq, cfg.Hkv, cfg.d
    g = _upload_prefill(inp, dev)
    sampler = ClockSampler(dev.index if world == 1 else local)
    sampler.start()
    ms, swa_ms, x_ms, o, oc, ws, err = time_prefill(g, cfg, dev, args.steps, warmup, world)
    clocks = sampler.stop()
    tokens = B * T
    nbytes = swa_bytes(B, T, Hq, Hkv, d)
    step_bytes = nbytes + xattn_bytes(inp.pos, Hq, Hkv, d, T)
    line = {
        "metric": METRIC, "value": tokens * world / (ms / 1e3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": _config_line(cfg),
        "roofline": step_roofline(nbytes, step_bytes, ms, peaks, cfg.name),
        "swa_alone": hbm_roofline("swa_tc", nbytes, swa_ms, peaks, f"swa_fwd_{cfg.name}", SWA_SOURCES),
        "step": {"algorithmic_bytes": step_bytes, "frac": step_bytes / (ms / 1e3) / 1e9 / peaks["hbm"],
                 "swa_alone_ms": swa_ms, "xattn_alone_ms": x_ms},
        "gpu_launches": args.steps * launches_per_prefill_step(cfg),
        "clocks": clocks,
    }
    if "e2e" in legs:
        line["e2e"] = run_e2e(g, o, oc, ws, err, inp, cfg, dev, args.steps, world)
    if "gradient" in legs:
        line["gradient"] = run_gradient(dev, world, g, o, oc, cfg, peaks)
    del g, o, oc, ws
    torch.cuda.empty_cache()
    if "decode" in legs:
        line["decode"] = run_decode(dev, world, peaks, "decode_128k")
    if "decode_b8" in legs:
        line["decode_b8"] = run_decode(dev, world, peaks, "decode_128k_b8")
    torch.cuda.empty_cache()
    if "sft" in legs:
        line["sft"] = run_sft(dev, world, peaks, max(5, min(args.steps, 20)), warmup)
        torch.cuda.empty_cache()
    if "prefill_1m" in legs:
        line["prefill_1m"] = run_prefill_1m(dev, world, peaks, max(3, min(args.steps, 10)), warmup)
        torch.cuda.empty_cache()
    if rank == 0:
        line["cpu_baseline"] = cpu_baselines(inp) if (world == 1 and "cpu" in legs) else None
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="orthros", choices=["orthros", "reference"])
    ap.add_argument("--config", default="prefill_128k", choices=["prefill_128k", "prefill_1m", "sft_16k",
                                                                 "tiny_prefill", "prefill_16k", "sft_16k_1"])
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch size (profiling)")
    ap.add_argument("--legs", default="", help=f"comma list of legs to run (default all: {','.join(ALL_LEGS)})")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
