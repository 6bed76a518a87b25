#!/usr/bin/env python
"""Benchmark of the fused RoPE + causal attention forward (prefill).

One step = one call of the whole hot path (attn_fwd) over one batch of the
workload, inputs resident on the device.  The `e2e` figure times the
host-buffer entry attn_fwd_host instead: inputs copied in from pinned host
memory and outputs copied back every step.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Metric: causal attention forward TFLOP/s, counting the useful causal QK^T and
PV work 2*B*Hq*S^2*D per step ("Flash Attention: Causal Prefill D=128",
Performance measurements: TFLOPS = 2*B*H*S*S*D / (ms*1e9)).  With N > 1
(torchrun) every rank runs its own independent batch of the same shape (the
path shards by batch and head with no exchange), `value` is the job total.

--impl reference times the float64 CPU oracle on the host cores instead, one
bounded sample of query rows per step, on the same metric.

Besides the contract's keys, each line of ours carries `timing_ms` (min, p10,
median, p90, max and count of the per-step CUDA-event times) and `source_sha`
(the hash of the CUDA and host sources that ran; the DRAM traffic records in
profiles/ are matched against it).  Other legs: --decode, --backward,
--blocksparse, --local (and --backward with either of the last two).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import seeded_inputs as si  # noqa: E402

METRIC = "causal attn fwd TFLOP/s at S=8192 D=128 bf16; % of GB300 dense BF16 peak"
DEFAULT_WORKLOAD = "rope_causal_s8192"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024


def useful_flops(w):
    return 2.0 * w["B"] * w["Hq"] * w["S"] * w["S"] * w["D"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_config(name, w):
    cfg = {"workload": name, "B": w["B"], "Hq": w["Hq"], "Hkv": w["Hkv"], "S": w["S"], "D": w["D"],
           "causal": w["causal"], "rope_base": w["rope_base"], "window_k": w["window_k"],
           "outlier_channels": w["outliers"], "layout": "BSHD", "inputs": "seeded iid N(0,1) bf16"}
    return cfg


# --------------------------------------------------------------------- CPU oracle timing
def time_oracle(q, k, v, w, budget_s, seed=si.MASTER_SEED):
    """Time the float64 oracle on a bounded sample of query rows; returns (TFLOP/s, seconds, sample, threads).

    Samples grow (more seeded rows, then further seeded sets of 8 heads) until
    about budget_s seconds of oracle time have been spent.
    """
    import oracle
    B, Hq, Hkv, S = w["B"], w["Hq"], w["Hkv"], w["S"]
    nrows = 4
    total_flops = 0.0
    total_time = 0.0
    rows_done = 0
    head_sets = 0
    while total_time < budget_s:
        heads = si.sample_heads(seed + 97 * head_sets, B, Hq, Hkv, 8)
        rows = si.sample_rows(seed + nrows, S, nrows)
        rb = np.repeat([b for b, _ in heads], len(rows))
        rh = np.repeat([h for _, h in heads], len(rows))
        ri = np.tile(rows, len(heads))
        t0 = time.perf_counter()
        oracle.attn_rows(q, k, v, rb, rh, ri, causal=w["causal"], rope_base=w["rope_base"],
                         window_k=w["window_k"])
        dt = time.perf_counter() - t0
        keys = (ri.astype(np.float64) + 1.0) if w["causal"] else np.full(len(ri), float(S))
        total_flops += float(np.sum(4.0 * w["D"] * keys))
        total_time += dt
        rows_done += len(ri)
        if nrows >= S:
            head_sets += 1  # every row of these heads done: continue with other heads
        else:
            nrows = min(S, max(nrows * 2, int(nrows * min(8.0, 0.5 * budget_s / max(dt, 1e-3)))))
    sample = (f"{rows_done} query rows over {head_sets + 1} seeded sets of {len(heads)} (batch, head) pairs, useful work "
              f"4*D*(keys) per row, {total_time:.1f} s")
    return total_flops / total_time / 1e12, total_time, sample, oracle.threads()


# --------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    # where the raw samples go: $ATTN_CLOCK_LOG_DIR if set (to keep them), else a temporary folder
    LOG_DIR = os.environ.get("ATTN_CLOCK_LOG_DIR") or os.path.join(tempfile.gettempdir(), "attn_bench_clocks")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join(self.LOG_DIR, f"clocks_gpu{index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------- replicas (N > 1)
# Every (batch, head) of the forward is independent: with N ranks each rank
# runs the whole workload on its own seeded batch (weak scaling, no
# collective on the data path); only the timings meet, as a max over ranks.
def replica_seed(rank):
    return si.MASTER_SEED + rank


def max_over_ranks(values, dist, device):
    """Element-wise maximum of a list of floats over all ranks (identity without a process group)."""
    import torch
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_tflops(world, flops_per_rank, ms):
    """Units all ranks processed / the slowest rank's time."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


# --------------------------------------------------------------------- our arm
def run_ours(args, w, rank, world, local_rank):
    import torch
    import attention_causal_attn_gb300 as attn

    attn.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    B, Hq, Hkv, S, D = w["B"], w["Hq"], w["Hkv"], w["S"], w["D"]
    seed = replica_seed(rank)  # every rank its own independent batch
    q_h, k_h, v_h = si.make_qkv(B, Hq, Hkv, S, D, outliers=w["outliers"], seed=seed)
    to_pinned = lambda a: torch.from_numpy(a).view(torch.bfloat16).pin_memory()
    q_p, k_p, v_p = to_pinned(q_h), to_pinned(k_h), to_pinned(v_h)
    q, k, v = q_p.to(dev), k_p.to(dev), v_p.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    kw = dict(causal=w["causal"], rope_base=w["rope_base"], window_k=w["window_k"], stream=stream)
    prerotate = args.rope_lowering == "prerotate"
    launches_per_step = 3 if prerotate else 1
    if prerotate:
        # the other side of the Rotation Calculus: rotate Q and K in their own pass, then
        # the attention without in-loop rotation (three launches per step)
        if not w["rope_base"] or w["window_k"]:
            raise SystemExit("--rope-lowering prerotate needs RoPE on and the window off")
        q_rot = torch.empty(q.shape, dtype=torch.float16, device=dev)
        k_rot = torch.empty(k.shape, dtype=torch.float16, device=dev)

        def step():
            attn.attn_rope_rotate(q, w["rope_base"], out=q_rot, stream=stream)
            attn.attn_rope_rotate(k, w["rope_base"], out=k_rot, stream=stream)
            attn.attn_fwd_rotated(q_rot, k_rot, v, o, lse, causal=w["causal"], stream=stream)
    else:
        def step():
            attn.attn_fwd(q, k, v, o, lse, **kw)

    for _ in range(max(args.warmup, 3)):
        step()
    attn.attn_check(stream=stream, device=dev)

    def barrier():
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # device-timed region: K back-to-back steps, events on the launching stream
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        barrier()
        t_begin.record(stream)
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        t_end.record(stream)
        barrier()
    attn.attn_check(stream=stream, device=dev)
    elapsed_ms = t_begin.elapsed_time(t_end)
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]

    # end-to-end through the C-ABI host-buffer entry (attn_fwd_host): every step copies
    # the inputs from pinned host memory and the outputs back, overlapped chunk by
    # chunk with the compute; the call returns with O and LSE in host memory, so the
    # host clock around the synchronous calls brackets the whole step
    o_h = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    hkw = dict(causal=w["causal"], rope_base=w["rope_base"], window_k=w["window_k"], device=dev)

    def e2e_step():
        attn.attn_fwd_host(q_p, k_p, v_p, o_h, lse_h, **hkw)

    for _ in range(2):
        e2e_step()
    barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_ms = (time.perf_counter() - t0) * 1e3 / e2e_steps
    barrier()

    elapsed_ms, e2e_ms, launch_avg_ms = max_over_ranks([elapsed_ms, e2e_ms, float(np.mean(launch_ms))], dist, dev)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        tf, secs, sample, threads = time_oracle(q_h, k_h, v_h, w, args.cpu_budget)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample}
        # the same oracle on one host core, a shorter sample
        import oracle
        oracle.set_threads(1)
        try:
            tf1, _, sample1, _ = time_oracle(q_h, k_h, v_h, w, max(1.0, args.cpu_budget / 4))
        finally:
            oracle.set_threads(threads)
        cpu["value_1core"] = tf1
        cpu["sample_1core"] = sample1
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return None

    flops = useful_flops(w)
    ms_per_step = elapsed_ms / args.steps
    value = whole_job_tflops(world, flops, ms_per_step)
    peaks, peak_kind = load_peaks()
    peak = float(peaks["bf16_tflops"])
    peak_sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    achieved = flops / (launch_avg_ms * 1e-3) / 1e12
    in_bytes = q.numel() * 2 + k.numel() * 2 + v.numel() * 2
    out_bytes = o.numel() * 2 + lse.numel() * 4
    cfg = workload_config(args.workload, w)
    cfg["rope_lowering"] = "pre-rotation pass + attention" if prerotate else "fused at load"
    cfg["l2"] = f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB of Q/K/V per step vs 129 MB L2), no flush"
    cfg["timing"] = f"CUDA events on the launching stream, {args.steps} steps after {max(args.warmup, 3)} warm-up"
    # the committed DRAM count belongs to the named workload at its own size, fused
    same_shape = args.batch is None and args.seq is None and args.window_k is None and not prerotate
    traffic = load_traffic(args.workload) if same_shape else None
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": cfg,
        "pct_of_peak": {"measured_bf16_burst": round(value / world / peak, 4),
                        "measured_bf16_sustained": round(value / world / peak_sustained, 4),
                        "peak_kind": peak_kind},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": ("step: 2 x rope_rotate_kernel + attn_fwd_kernel" if prerotate else "attn_fwd_kernel"),
                     "peak_source": f"bf16_tflops ({peak_kind}, burst)",
                     "algorithmic": "2*B*Hq*S^2*D useful causal FLOPs per launch"},
        "cpu_baseline": cpu,
        "e2e": {"value": round(whole_job_tflops(world, flops, e2e_ms), 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes,
                "ms_per_step": round(e2e_ms, 4), "entry": "attn_fwd_host (RoPE fused at load)"},
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clocks.summary(),
        "timing_ms": timing_stats(launch_ms),
    }
    return line


def timing_stats(samples_ms):
    """min / p10 / median / p90 / max of the per-step CUDA-event times (ms) and their count."""
    a = np.asarray(samples_ms, dtype=np.float64)
    q = np.percentile(a, [0, 10, 50, 90, 100])
    return {"n": int(a.size), "min": round(float(q[0]), 4), "p10": round(float(q[1]), 4),
            "median": round(float(q[2]), 4), "p90": round(float(q[3]), 4), "max": round(float(q[4]), 4)}


def load_traffic(workload, kernel="attn_fwd_kernel"):
    """DRAM bytes per launch from the committed ncu summary of this kernel and workload, if present."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        if d.get("kernel_source_sha") == kernel_source_sha():
            return d.get("dram_bytes_per_launch")
    return None


def same_shape(args):
    """True when the run keeps the workload's own shape (no batch or length override)."""
    return args.batch is None and args.seq is None


def kernel_source_sha():
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_causal_attn_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        if fn.endswith((".cu", ".cuh", ".inc", ".h", ".cpp")):
            with open(os.path.join(csrc, fn), "rb") as f:
                h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


# --------------------------------------------------------------------- decode
def decode_bytes(w):
    """K/V bytes a decode step must read: V whole, K without the 16-byte pair chunks the window skips."""
    import attention_causal_attn_gb300 as attn
    B, Hkv, S, D = w["B"], w["Hkv"], w["S"], w["D"]
    v_bytes = B * S * Hkv * D * 2
    if not w["window_k"]:
        return 2 * v_bytes
    _, _, win = attn.attn_build_tables(1, D, w["rope_base"], w["window_k"])
    dist = np.arange(S - 1, -1, -1, dtype=np.int64)  # key j sits at distance S-1-j
    cut = np.searchsorted(win.astype(np.int64), dist, side="left")  # pairs with W_r < dist
    kept_chunks = (D // 2 - (cut // 8) * 8) * 2  # channels loaded per key (whole 8-pair chunks skipped)
    return v_bytes + int(B * Hkv * 2 * kept_chunks.sum())


def set_l2_fetch_granularity(nbytes):
    """Set this process's CUDA context hint for the DRAM fetch size behind an L2 miss
    (cudaLimitMaxL2FetchGranularity, 0..128 bytes).  It ends with the process; nothing on the
    GPU outlives it.  Returns (before, after) in bytes."""
    import ctypes
    rt = None
    for name in ("libcudart.so.13", "libcudart.so"):
        try:
            rt = ctypes.CDLL(name)
            break
        except OSError:
            continue
    if rt is None:
        raise RuntimeError("the CUDA runtime library was not found")
    limit = 5  # cudaLimitMaxL2FetchGranularity
    before, after = ctypes.c_size_t(0), ctypes.c_size_t(0)
    if rt.cudaDeviceGetLimit(ctypes.byref(before), limit) != 0:
        raise RuntimeError("cudaDeviceGetLimit(cudaLimitMaxL2FetchGranularity) failed")
    if rt.cudaDeviceSetLimit(limit, ctypes.c_size_t(nbytes)) != 0:
        raise RuntimeError("cudaDeviceSetLimit(cudaLimitMaxL2FetchGranularity) failed")
    rt.cudaDeviceGetLimit(ctypes.byref(after), limit)
    return before.value, after.value


def run_decode(args, w, rank, world, local_rank):
    """One step = one attn_decode call (the newest token of each sequence against its cache)."""
    import torch
    import attention_causal_attn_gb300 as attn
    attn.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    B, Hq, Hkv, S, D = w["B"], w["Hq"], w["Hkv"], w["S"], w["D"]
    q_full, k_h, v_h = si.make_qkv(B, 1, Hkv, S, D, seed=replica_seed(rank))
    q_h = si.bshd_bf16(replica_seed(rank), 4, B, 1, Hq, D)[:, 0]
    k, v = (torch.from_numpy(x).view(torch.bfloat16).to(dev) for x in (k_h, v_h))
    q = torch.from_numpy(np.ascontiguousarray(q_h)).view(torch.bfloat16).to(dev)
    fetch = set_l2_fetch_granularity(args.l2_fetch_bytes) if args.l2_fetch_bytes is not None else None
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(args.warmup, 3)):
        attn.attn_decode(q, k, v, o, lse, rope_base=w["rope_base"], window_k=w["window_k"], stream=stream)
    attn.attn_check(stream=stream, device=dev)
    # caches larger than L2 are streamed from HBM on every step; smaller ones get an L2 flush between steps
    kv_bytes = 2 * k.numel() * 2
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if kv_bytes < (256 << 20) else None
    times = []
    with ClockSampler(local_rank) as clocks:
        for _ in range(args.steps):
            if flush is not None:
                flush.fill_(1)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            attn.attn_decode(q, k, v, o, lse, rope_base=w["rope_base"], window_k=w["window_k"], stream=stream)
            e1.record(stream)
            times.append((e0, e1))
        torch.cuda.synchronize(dev)
    attn.attn_check(stream=stream, device=dev)
    step_ms = [a.elapsed_time(b) for a, b in times]
    ms = float(np.median(step_ms))
    same_shape = args.batch is None and args.seq is None and args.window_k is None and args.l2_fetch_bytes is None
    nbytes = decode_bytes(w)
    peaks, peak_kind = load_peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    cfg = workload_config(args.workload, w)
    cfg["step"] = "decode: one query per sequence at position S-1 against the whole cache"
    cfg["l2"] = "cache larger than L2, streamed every step" if flush is None else "L2 flushed between steps"
    if fetch is not None:
        cfg["l2_fetch_granularity_bytes"] = {"before": fetch[0], "during": fetch[1]}
    return {
        "metric": "decode K/V read GB/s", "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg,
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                     "frac": round(gbs / float(peaks["hbm_gbs"]), 4),
                     "traffic": load_traffic(args.workload, "decode_split_kernel") if same_shape else None,
                     "kernel": "decode_split_kernel + decode_combine_kernel",
                     "algorithmic": "K/V bytes read per step (window-skipped K chunks excluded), median step time"},
        "gpu_launches": 2 * args.steps, "clocks": clocks.summary(), "timing_ms": timing_stats(step_ms),
    }


# --------------------------------------------------------------------- backward
def run_backward(args, w, rank, world, local_rank):
    """One step = one attn_bwd call (dO.O rows, dK/dV, dQ) on the forward's own O and LSE."""
    import torch
    import attention_causal_attn_gb300 as attn
    attn.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if w["window_k"]:
        raise SystemExit("the backward has no window: pass --window-k 0")
    B, Hq, Hkv, S, D = w["B"], w["Hq"], w["Hkv"], w["S"], w["D"]
    q_h, k_h, v_h = si.make_qkv(B, Hq, Hkv, S, D, outliers=w["outliers"], seed=replica_seed(rank))
    do_h = si.bshd_bf16(replica_seed(rank), 9, B, S, Hq, D)
    q, k, v, dO = (torch.from_numpy(x).view(torch.bfloat16).to(dev) for x in (q_h, k_h, v_h, do_h))
    stream = torch.cuda.current_stream(dev)
    kw = dict(causal=w["causal"], rope_base=w["rope_base"], stream=stream)
    mask = None
    local = None
    if args.local:  # the backward of the sliding-window / ALiBi forward
        if "local" not in w:
            raise SystemExit("--local needs a workload with a window or ALiBi (sliding_window_s4096, alibi_s4096)")
        local = (w["local"]["window"], w["local"]["alibi"])
        kw.update(window=local[0], alibi=local[1])
        o, lse = attn.attn_fwd_local(q, k, v, **kw)
    elif args.blocksparse:  # the backward of the block-sparse forward, over the workload's mask
        if "block_mask" not in w:
            raise SystemExit("--blocksparse needs a workload with a block mask (bigbird_s4096)")
        mask = si.bigbird_block_mask(S, causal=w["causal"], **w["block_mask"])
        o, lse = attn.attn_fwd_blocksparse(q, k, v, *mask, **kw)
        kw["block_mask"] = mask
    else:
        o, lse = attn.attn_fwd(q, k, v, **kw)
    bwd = attn.attn_bwd_local if local is not None else attn.attn_bwd
    for _ in range(max(args.warmup, 3)):
        bwd(q, k, v, o, lse, dO, **kw)
    attn.attn_check(stream=stream, device=dev)
    times = []
    with ClockSampler(local_rank) as clocks:
        for _ in range(args.steps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            bwd(q, k, v, o, lse, dO, **kw)
            e1.record(stream)
            times.append((e0, e1))
        torch.cuda.synchronize(dev)
    attn.attn_check(stream=stream, device=dev)
    step_ms = [a.elapsed_time(b) for a, b in times]
    ms = float(np.median(step_ms))
    # useful backward work: 2.5 x the forward's 4*D FLOPs per visible (query, key) pair (dV, dP, dQ, dK
    # and the recomputed S); the kernels execute 7/5 of it, S and dP being formed in both tile kernels
    if local is not None:
        pairs = local_pairs(S, w["causal"], local[0])
    elif mask is not None:
        pairs = visible_pairs(S, *mask, w["causal"])
    else:
        pairs = S * S * (0.5 if w["causal"] else 1.0)
    flops = 2.5 * 4.0 * D * pairs * B * Hq
    tf = flops / (ms * 1e-3) / 1e12
    peaks, _ = load_peaks()
    cfg = workload_config(args.workload, w)
    cfg["step"] = "backward: dO.O rows, dK/dV kernel, dQ kernel on the forward's O and LSE"
    if mask is not None:
        cfg["step"] += ", over the block mask"
        cfg["active_blocks"] = int(mask[0][-1])
    if local is not None:
        cfg["step"] += ", with the sliding window / ALiBi bias"
        cfg["window"], cfg["alibi"] = local
    cfg["l2"] = "inputs larger than L2" if 4 * q.numel() * 2 > (256 << 20) else "inputs may stay in L2 between steps"
    return {
        "metric": "attention backward TFLOP/s", "value": round(tf, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg,
        "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": float(peaks["bf16_tflops"]),
                     "unit": "TFLOP/s", "frac": round(tf / float(peaks["bf16_tflops"]), 4), "traffic": None,
                     "kernel": ("bwd_dot_kernel + 2 x rope_rotate_kernel + bwd_dkdv_kernel + bwd_dq_kernel"
                                if w["rope_base"] else "bwd_dot_kernel + bwd_dkdv_kernel + bwd_dq_kernel"),
                     "algorithmic": "10*D FLOPs per visible (query, key) pair and head (2.5 x the forward's), "
                                    "median step time"},
        # the row reduction, the dK/dV and dQ kernels, and with RoPE the two rotation passes
        "gpu_launches": (5 if w["rope_base"] else 3) * args.steps, "clocks": clocks.summary(),
        "timing_ms": timing_stats(step_ms),
    }


# --------------------------------------------------------------------- block-sparse forward
def visible_pairs(S, row_ptr, col_idx, causal, block=128):
    """(query, key) pairs a block mask leaves visible: each listed block's rows x keys, triangular on the diagonal."""
    total = 0
    for r in range(len(row_ptr) - 1):
        rows = min(block, S - block * r)
        for c in col_idx[row_ptr[r]:row_ptr[r + 1]]:
            keys = min(block, S - block * int(c))
            if causal and int(c) == r:
                total += rows * (rows + 1) // 2
            else:
                total += rows * keys
    return total


def run_blocksparse(args, w, rank, world, local_rank):
    """One step = one attn_fwd_blocksparse call over the workload's block mask."""
    import torch
    import attention_causal_attn_gb300 as attn
    attn.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if "block_mask" not in w:
        raise SystemExit("--blocksparse needs a workload with a block mask (bigbird_s4096)")
    B, Hq, Hkv, S, D = w["B"], w["Hq"], w["Hkv"], w["S"], w["D"]
    q_h, k_h, v_h = si.make_qkv(B, Hq, Hkv, S, D, outliers=w["outliers"], seed=replica_seed(rank))
    rp, ci = si.bigbird_block_mask(S, causal=w["causal"], **w["block_mask"])
    q, k, v = (torch.from_numpy(x).view(torch.bfloat16).to(dev) for x in (q_h, k_h, v_h))
    stream = torch.cuda.current_stream(dev)
    kw = dict(causal=w["causal"], rope_base=w["rope_base"], stream=stream)
    o, lse = attn.attn_fwd_blocksparse(q, k, v, rp, ci, **kw)
    for _ in range(max(args.warmup, 3)):
        attn.attn_fwd_blocksparse(q, k, v, rp, ci, o, lse, **kw)
    attn.attn_check(stream=stream, device=dev)
    small = 3 * q.numel() * 2 < (256 << 20)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if small else None
    times = []
    with ClockSampler(local_rank) as clocks:
        for _ in range(args.steps):
            if flush is not None:
                flush.fill_(1)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            attn.attn_fwd_blocksparse(q, k, v, rp, ci, o, lse, **kw)
            e1.record(stream)
            times.append((e0, e1))
        torch.cuda.synchronize(dev)
    attn.attn_check(stream=stream, device=dev)
    step_ms = [a.elapsed_time(b) for a, b in times]
    ms = float(np.median(step_ms))
    pairs = visible_pairs(S, rp, ci, w["causal"])
    flops = 4.0 * D * pairs * B * Hq
    tf = flops / (ms * 1e-3) / 1e12
    peaks, _ = load_peaks()
    nb = len(rp) - 1
    cfg = workload_config(args.workload, w)
    cfg["step"] = "block-sparse forward over the workload's mask"
    cfg["active_blocks"] = int(rp[-1])
    cfg["active_share"] = round(int(rp[-1]) / (nb * nb), 4)
    cfg["l2"] = "L2 flushed between steps" if flush is not None else "inputs larger than L2"
    return {
        "metric": "block-sparse attention forward TFLOP/s", "value": round(tf, 2), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": cfg,
        "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": float(peaks["bf16_tflops"]),
                     "unit": "TFLOP/s", "frac": round(tf / float(peaks["bf16_tflops"]), 4),
                     "traffic": load_traffic(args.workload, "bs_fwd_kernel") if same_shape(args) else None,
                     "kernel": "bs_fwd_kernel",
                     "algorithmic": "4*D FLOPs per visible (query, key) pair of the mask, median step time"},
        "gpu_launches": args.steps, "clocks": clocks.summary(), "timing_ms": timing_stats(step_ms),
    }


# --------------------------------------------------------------------- sliding window / ALiBi
def local_pairs(S, causal, win):
    """Visible (query, key) pairs under the sliding window |i - j| < win (win 0: none) and the causal mask."""
    i = np.arange(S, dtype=np.int64)
    if causal:
        return int(np.minimum(i + 1, win).sum()) if win else S * (S + 1) // 2
    return int((np.minimum(i + win, S) - np.maximum(i - win + 1, 0)).sum()) if win else S * S


def run_local(args, w, rank, world, local_rank):
    """One step = one attn_fwd_local call (sliding window and/or ALiBi) on the workload."""
    import torch
    import attention_causal_attn_gb300 as attn
    attn.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if "local" not in w:
        raise SystemExit("--local needs a workload with a window or ALiBi (sliding_window_s4096, alibi_s4096)")
    B, Hq, Hkv, S, D = w["B"], w["Hq"], w["Hkv"], w["S"], w["D"]
    win, alibi = w["local"]["window"], w["local"]["alibi"]
    q_h, k_h, v_h = si.make_qkv(B, Hq, Hkv, S, D, outliers=w["outliers"], seed=replica_seed(rank))
    q, k, v = (torch.from_numpy(x).view(torch.bfloat16).to(dev) for x in (q_h, k_h, v_h))
    stream = torch.cuda.current_stream(dev)
    kw = dict(causal=w["causal"], rope_base=w["rope_base"], window=win, alibi=alibi, stream=stream)
    o, lse = attn.attn_fwd_local(q, k, v, **kw)
    for _ in range(max(args.warmup, 3)):
        attn.attn_fwd_local(q, k, v, o, lse, **kw)
    attn.attn_check(stream=stream, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if 3 * q.numel() * 2 < (256 << 20) else None
    times = []
    with ClockSampler(local_rank) as clocks:
        for _ in range(args.steps):
            if flush is not None:
                flush.fill_(1)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            attn.attn_fwd_local(q, k, v, o, lse, **kw)
            e1.record(stream)
            times.append((e0, e1))
        torch.cuda.synchronize(dev)
    attn.attn_check(stream=stream, device=dev)
    step_ms = [a.elapsed_time(b) for a, b in times]
    ms = float(np.median(step_ms))
    tf = 4.0 * D * local_pairs(S, w["causal"], win) * B * Hq / (ms * 1e-3) / 1e12
    peaks, _ = load_peaks()
    cfg = workload_config(args.workload, w)
    cfg["step"] = "forward with the sliding window / ALiBi bias"
    cfg["window"], cfg["alibi"] = win, alibi
    cfg["l2"] = "L2 flushed between steps" if flush is not None else "inputs larger than L2"
    return {
        "metric": "local attention forward TFLOP/s", "value": round(tf, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg,
        "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": float(peaks["bf16_tflops"]),
                     "unit": "TFLOP/s", "frac": round(tf / float(peaks["bf16_tflops"]), 4),
                     "traffic": load_traffic(args.workload, "bs_fwd_kernel") if same_shape(args) else None,
                     "kernel": "bs_fwd_kernel (EXT)",
                     "algorithmic": "4*D FLOPs per visible (query, key) pair, median step time"},
        "gpu_launches": args.steps, "clocks": clocks.summary(), "timing_ms": timing_stats(step_ms),
    }


# --------------------------------------------------------------------- reference arm
def run_reference(args, w, rank):
    if rank != 0:
        return None
    q_h, k_h, v_h = si.make_qkv(w["B"], w["Hq"], w["Hkv"], w["S"], w["D"], outliers=w["outliers"])
    per_step = max(0.5, args.ref_budget / max(1, args.steps + args.warmup))
    for i in range(args.warmup):
        time_oracle(q_h, k_h, v_h, w, per_step, seed=si.MASTER_SEED + 1000 + i)
    vals, secs, sample, threads = [], 0.0, "", 1
    for i in range(args.steps):
        tf, s, sample, threads = time_oracle(q_h, k_h, v_h, w, per_step, seed=si.MASTER_SEED + i)
        vals.append(tf)
        secs += s
    value = float(np.mean(vals))
    flops = useful_flops(w)
    cfg = workload_config(args.workload, w)
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": args.gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": flops / (value * 1e12) * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": cfg,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"per step: {sample}; ms_per_step extrapolated from the sampled rate"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(si.WORKLOADS))
    ap.add_argument("--window-k", type=float, default=None, help="override the workload's window multiplier")
    ap.add_argument("--batch", type=int, default=None, help="override the workload's batch (profiling captures)")
    ap.add_argument("--seq", type=int, default=None, help="override the workload's sequence length")
    ap.add_argument("--decode", action="store_true",
                    help="time one decode step (attn_decode) on the workload's cache shape instead of the prefill")
    ap.add_argument("--local", action="store_true",
                    help="time the sliding-window / ALiBi forward (sliding_window_s4096, alibi_s4096); "
                         "with --backward, its backward")
    ap.add_argument("--blocksparse", action="store_true",
                    help="time the block-sparse forward on a workload with a block mask (bigbird_s4096)")
    ap.add_argument("--backward", action="store_true",
                    help="time one backward step (attn_bwd) on the workload instead of the forward")
    ap.add_argument("--l2-fetch-bytes", type=int, default=None,
                    help="decode only: set the context's L2 fetch granularity hint (32 lets the window's "
                         "skipped 16-byte K chunks stay unread in DRAM)")
    ap.add_argument("--rope-lowering", default="fused", choices=["fused", "prerotate"],
                    help="fused: RoPE at load (the specified path); prerotate: a rotation pass, then the attention")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=90.0, help="seconds of oracle time for --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    w = dict(si.WORKLOADS[args.workload])
    if args.window_k is not None:
        w["window_k"] = args.window_k if args.window_k > 0 else None
    if args.batch is not None:
        w["B"] = args.batch
    if args.seq is not None:
        w["S"] = args.seq
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, w, rank)
    elif args.decode:
        line = run_decode(args, w, rank, world, local_rank)
    elif args.backward:
        line = run_backward(args, w, rank, world, local_rank)
    elif args.local:
        line = run_local(args, w, rank, world, local_rank)
    elif args.blocksparse:  # forward; with --backward the branch above times its backward
        line = run_blocksparse(args, w, rank, world, local_rank)
    else:
        line = run_ours(args, w, rank, world, local_rank)
    if line is not None:
        if args.impl != "reference":
            line["source_sha"] = kernel_source_sha()  # hash of the CUDA and host sources that ran
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
