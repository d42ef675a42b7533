"""Benchmark of the Orthros per-layer attention operator on GB300.

Default workload: 8B-class prefill, batch 2 x 131072 tokens, 32 query heads /
8 KV heads, d=128, w=128, one output copy per sequence at its last position.
One step = base SWA (Eq. 4) over every token + the copies' cross-attention
(Eq. 5), i.e. the whole prefill hot path.  The line also reports decode steps/s
(batch 2, 131072-token cache, 128 consecutive fused decode steps) and the time of
the base stream's gradient (orthros_swa_bwd) on the prefill inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl orthros|reference]

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

from synthetic import CONFIGS, SEEDS, make_decode, make_prefill  # noqa: E402

METRIC = "prefill tokens/s (SWA+1 global query) at 128K; decode steps/s; % of HBM peak"
KERNEL_SRC = os.path.join(ROOT, "long_context_attention_orthros_gb300", "csrc")


# ----------------------------------------------------------------- helpers

def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def kernel_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(KERNEL_SRC, n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _profile_traffic(name, src_hash):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", f"{name}.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("kernel_source_sha256_16") != src_hash:
        return None
    return d.get("dram_bytes_per_launch")


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


# ----------------------------------------------------------------- CPU oracle baseline

def oracle_prefill_rate(inp, target_s: float = 8.0):
    """The fp64 oracle on a bounded sample of the prefill workload: base rows in the
    middle of each sequence (all heads) plus the copies' full cross-attention.
    Returns (tokens/s, threads, sample description)."""
    import oracle
    cfg = inp.cfg
    q = inp.q_base
    t_x0 = time.perf_counter()
    oracle.xattn(np.ascontiguousarray(inp.qc_raw), inp.pos, inp.k, inp.v, inp.alpha_c, inp.beta_c, cfg.scale)
    t_x = time.perf_counter() - t_x0
    n = 256
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
    per_token = dt / n + t_x / (cfg.B * cfg.T)
    sample = (f"{n} base tokens x {cfg.Hq} heads (fp64 SWA rows) + {cfg.B * cfg.T_out} copies over "
              f"{cfg.T} keys; {dt + t_x:.1f} s wall")
    return 1.0 / per_token, oracle.num_threads(), sample


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    cfg = CONFIGS[args.config]
    inp = make_prefill(cfg, SEEDS[cfg.name])
    import oracle
    oracle.build()
    rates, descs = [], ""
    for i in range(args.warmup + args.steps):
        r, threads, descs = oracle_prefill_rate(inp, target_s=4.0)
        if i >= args.warmup:
            rates.append(r)
    value = statistics.mean(rates)
    tokens = cfg.B * cfg.T
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tokens / value * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": cfg.name, "B": cfg.B, "T": cfg.T, "Hq": cfg.Hq,
                                        "Hkv": cfg.Hkv, "d": cfg.d, "window": cfg.window, "T_out": cfg.T_out},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": descs},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- GPU arm

def run_gpu(args):
    import torch
    import long_context_attention_orthros_gb300 as orth

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    hbm_peak, _tf_peak, peak_kind = _peaks()

    cfg = CONFIGS[args.config]
    inp = make_prefill(cfg, SEEDS[cfg.name] + 1000 * rank)
    B, T, Hq, Hkv, d, T_out = cfg.B, cfg.T, cfg.Hq, cfg.Hkv, cfg.d, cfg.T_out

    def pinned(x, dtype):
        t = torch.empty(x.shape, dtype=dtype, pin_memory=True)
        t.numpy()[...] = x.view(np.int16) if dtype == torch.int16 else x
        return t

    h = {  # pinned host copies (the e2e arm copies these every step)
        "q": pinned(inp.q_raw, torch.int16), "k": pinned(inp.k, torch.int16),
        "v": pinned(inp.v, torch.int16), "qc": pinned(np.ascontiguousarray(inp.qc_raw), torch.int16),
        "pos": pinned(inp.pos, torch.int32), "a": pinned(inp.alpha, torch.float32),
        "b": pinned(inp.beta, torch.float32), "ac": pinned(inp.alpha_c, torch.float32),
        "bc": pinned(inp.beta_c, torch.float32),
    }
    g = {key: t.to(dev) for key, t in h.items()}
    for key in ("q", "k", "v", "qc"):
        g[key] = g[key].view(torch.bfloat16)
    o = torch.empty((B, T, Hq, d), dtype=torch.bfloat16, device=dev)
    oc = torch.empty((B, T_out, Hq, d), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(orth.xattn_workspace_size(B, T_out, T, Hq, Hkv, d), 256), dtype=torch.uint8,
                     device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ho = torch.empty((B, T, Hq, d), dtype=torch.int16, pin_memory=True)
    hoc = torch.empty((B, T_out, Hq, d), dtype=torch.int16, pin_memory=True)
    stream = torch.cuda.current_stream(dev)
    ev = []

    def step(timed_swa=False):
        if timed_swa:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
        orth.swa_fwd(g["q"], g["k"], g["v"], g["a"], g["b"], window=cfg.window, scale=cfg.scale,
                     out=o, dev_err=err)
        if timed_swa:
            e1.record(stream)
            ev.append((e0, e1))
        orth.xattn_fwd(g["qc"], g["pos"], g["k"], g["v"], g["ac"], g["bc"], scale=cfg.scale, out=oc,
                       workspace=ws, dev_err=err)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    sampler = ClockSampler(dev.index if world == 1 else local)
    sampler.start()
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step(timed_swa=True)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    ms = t0.elapsed_time(t1) / args.steps
    ms = allreduce_max(ms, world)
    swa_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    assert int(err.item()) == 0, f"device error word {int(err.item())}"

    tokens = B * T
    value = tokens * world / (ms / 1e3)
    swa_bytes = B * T * (2 * Hq + 2 * Hkv) * d * 2  # Q + O (Hq heads) + K + V, once each
    swa_gbs = swa_bytes / (swa_ms / 1e3) / 1e9
    swa_hash = kernel_hash("swa_fwd.cu", "swa_tc.cu", "tc.cuh", "common.cuh", "kernels.cuh")
    traffic = _profile_traffic(f"swa_fwd_{cfg.name}", swa_hash)

    # ---- end to end: pinned host inputs -> device -> kernels -> host outputs
    h2d = sum(h[k_].numel() * h[k_].element_size() for k_ in h)
    d2h = ho.numel() * 2 + hoc.numel() * 2

    # pipelined by 8K-row chunks on three streams: the upload of chunk c+1, the SWA of chunk c
    # (orthros_swa_fwd_rows; its key halo is in chunk c-1) and the download of chunk c-1 overlap;
    # the copies' cross-attention runs once the last K/V chunk is on the device
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

    e2e_steps = max(3, min(args.steps, 10))
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    a1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = allreduce_max(a0.elapsed_time(a1) / e2e_steps, world)

    # ---- decode: batch 2, 131072-token cache, 128 fused steps
    dec = None
    if not args.no_decode:
        dec = run_decode(args, dev, world, hbm_peak, peak_kind)

    # ---- base-stream gradient on the same inputs (training modes)
    bwd = None
    if not args.no_bwd:
        bwd = run_bwd(dev, world, g, o, oc, cfg, _tf_peak, peak_kind)

    del g, o, oc, ws
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": cfg.name, "B": B, "T": T, "Hq": Hq, "Hkv": Hkv, "d": d,
                   "window": cfg.window, "T_out": T_out,
                   "l2": f"inputs larger than L2 ({swa_bytes / 1e9:.1f} GB per step), no flush"},
        "roofline": {"kernel": "swa_fwd", "bound": "hbm", "achieved": swa_gbs, "peak": hbm_peak,
                     "unit": "GB/s", "frac": swa_gbs / hbm_peak, "traffic": traffic,
                     "peak_kind": peak_kind, "algorithmic_bytes": swa_bytes, "ms_per_launch": swa_ms},
        "e2e": {"value": tokens * world / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": args.steps * launches_per_prefill_step(cfg),
        "clocks": clocks,
        "decode": dec,
        "gradient": bwd,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r, threads, sample = oracle_prefill_rate(inp)
        line["cpu_baseline"] = {"value": r, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                "sample": sample}
    elif rank == 0:
        line["cpu_baseline"] = None
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def launches_per_prefill_step(cfg) -> int:
    """Kernels one prefill step launches: SWA, the copies' partial kernel, and the
    combine kernel unless each copy row has a single partial."""
    import long_context_attention_orthros_gb300 as orth  # noqa: F401  (library must exist)
    G = cfg.Hq // cfg.Hkv
    rows = cfg.T_out * G
    wk = 4 if rows <= 16 else 1
    # mirror of the split plan in xattn_fwd.cu (a single partial -> no combine launch)
    row_tiles = math.ceil(rows / (16 * (4 // wk)))
    base = cfg.B * cfg.Hkv * row_tiles
    splits = min(max(1, math.ceil(304 / base)), math.ceil(cfg.T / 256))
    chunk = math.ceil(math.ceil(cfg.T / splits) / 64) * 64
    splits = math.ceil(cfg.T / chunk)
    return 2 + (0 if splits * wk == 1 else 1)


def swa_pairs(B, T, Hq, w) -> int:
    """(query row, key) pairs of Eq. (4): row t sees min(t + 1, w) keys."""
    n = min(T, w)
    return B * Hq * (n * (n + 1) // 2 + (T - n) * w)


def run_bwd(dev, world, g, o, oc, cfg, tf_peak, peak_kind, calls: int = 5):
    """The layer's attention gradient on the prefill inputs with seeded N(0, 1) output
    gradients: orthros_attn_bwd, both streams in one call (each with its forward's
    log-sum-exp, computed untimed beforehand)."""
    import torch
    import long_context_attention_orthros_gb300 as orth
    B, T, Hq, Hkv, d, T_out = cfg.B, cfg.T, cfg.Hq, cfg.Hkv, cfg.d, cfg.T_out
    gen = torch.Generator(device=dev)
    gen.manual_seed(SEEDS[cfg.name] + 17)
    dO = torch.randn((B, T, Hq, d), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
    dOc = torch.randn((B, T_out, Hq, d), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
    ws = torch.empty(orth.attn_bwd_workspace_size(B, T, T_out, Hq, Hkv, d), dtype=torch.uint8, device=dev)
    qc = g["qc"].contiguous()
    q = g["q"] if g["q"].shape[1] == T else g["q"][:, :T].contiguous()  # appended copies: base rows only
    stream = torch.cuda.current_stream(dev)
    # a training forward keeps each row's log-sum-exp (both streams); the gradient takes it
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
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(calls):
        grads = call()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = allreduce_max(e0.elapsed_time(e1) / calls, world)
    assert all(bool(torch.isfinite(t).all()) for t in grads)
    del grads, dO, dOc, ws, lse, lsec, q
    # launches per call (mirror of attn_bwd.cu): fp16 K; base stream with its log-sum-exp: fp16 q,
    # D, dq, the dalpha / dbeta sums; copies with theirs: fp16 q, D, dq (one pass, or split over
    # the keys when one row tile per (batch, KV head) holds all copies); one dk/dv for both
    per_call = 1 + 4 + (3 if T_out > 0 else 0) + 1
    # the five contractions of the gradient (S, dP, dV, dK, dQ), 2 d flops each per pair
    pos = g["pos"].cpu().numpy().astype(np.int64)
    pairs = swa_pairs(B, T, Hq, cfg.window) + Hq * int((pos + 1).sum())
    flops = 10 * d * pairs
    tfs = flops / (ms / 1e3) / 1e12
    return {"value": B * T * world / (ms / 1e3), "unit": "tokens/s", "ms_per_call": ms,
            "what": "attn_bwd: both streams' gradient in one call (dK/dV written once), each stream with its "
                    "forward's log-sum-exp",
            "roofline": {"kernel": f"attn_bwd ({per_call} launches)", "bound": "tensor", "achieved": tfs,
                         "peak": tf_peak, "unit": "TFLOP/s", "frac": tfs / tf_peak, "traffic": None,
                         "peak_kind": peak_kind, "algorithmic_flops": flops},
            "gpu_launches": per_call * calls}


def run_decode(args, dev, world, hbm_peak, peak_kind):
    import torch
    import long_context_attention_orthros_gb300 as orth
    cfg = CONFIGS["decode_128k"]
    inp = make_decode(cfg, SEEDS[cfg.name])
    B, Hq, Hkv, d, S = cfg.B, cfg.Hq, cfg.Hkv, cfg.d, cfg.steps

    def bf(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(dev)

    kc, vc = bf(inp.k_cache), bf(inp.v_cache)
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

    cl.copy_(cl0)
    run_all()  # warm-up pass
    reps = 3
    total = 0.0
    for _ in range(reps):
        cl.copy_(cl0)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run_all()
        e1.record(stream)
        torch.cuda.synchronize()
        total += e0.elapsed_time(e1)
    assert int(err.item()) == 0, f"decode device error {int(err.item())}"
    ms_step = allreduce_max(total / (reps * S), world)
    # the same S steps captured once as a CUDA graph and replayed (no per-step launch from the host)
    graph = torch.cuda.CUDAGraph()
    cl.copy_(cl0)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        run_all()
    gtotal = 0.0
    for _ in range(reps):
        cl.copy_(cl0)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        gtotal += e0.elapsed_time(e1)
    assert int(err.item()) == 0, f"decode device error {int(err.item())} (graph)"
    gms_step = allreduce_max(gtotal / (reps * S), world)
    avg_len = cfg.T0 + (S + 1) / 2
    step_bytes = B * avg_len * Hkv * d * 2 * 2  # the whole cache's K and V, once per step
    gbs = step_bytes / (ms_step / 1e3) / 1e9
    return {"value": world / (ms_step / 1e3), "unit": "steps/s", "ms_per_step": ms_step,
            "config": {"workload": cfg.name, "B": B, "cache_len": cfg.T0, "steps": S, "Hq": Hq,
                       "Hkv": Hkv, "d": d, "window": cfg.window},
            "roofline": {"kernel": "decode_step", "bound": "hbm", "achieved": gbs, "peak": hbm_peak,
                         "unit": "GB/s", "frac": gbs / hbm_peak, "traffic": None,
                         "peak_kind": peak_kind, "algorithmic_bytes": step_bytes},
            "cuda_graph": {"value": world / (gms_step / 1e3), "unit": "steps/s", "ms_per_step": gms_step,
                           "note": f"the {S} steps captured once and replayed"},
            "gpu_launches": 2 * reps * S}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="orthros", choices=["orthros", "reference"])
    ap.add_argument("--config", default="prefill_128k", choices=["prefill_128k", "prefill_1m", "sft_16k",
                                                                 "tiny_prefill", "prefill_16k", "sft_16k_1"])
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-bwd", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
