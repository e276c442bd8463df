"""Benchmark: attention forward TFLOP/s on one GB300 (and % of dense bf16 peak).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--pass forward|backward]

One step = one fa_fwd launch over the whole workload (every batch, head and
query tile), inputs already resident in HBM.  TFLOP/s counts 4*D flops per
unmasked (query, key) pair.  Between timed steps the inputs rotate over enough
copies that their total exceeds twice the L2 cache.

Prints ONE JSON line (rank 0).  Besides the device-timed value it reports:
  e2e          the same metric through the public host-buffer call
               (attention_from_host: pinned host Q, K, V in, host O, LSE out; the
               copies and kernels overlap by chunks of heads) with every copy inside
               the timed region;
  roofline     achieved TFLOP/s of the kernel against the measured bf16 peak;
  cpu_baseline the fp64 oracle timed on the host cores on a bounded row sample;
  clocks       SM clocks and throttle reasons sampled during the timed region.
With --impl reference the fp64 CPU oracle is the measured arm (bounded row
samples of the same workload per step), printed with "impl": "reference".

Multi-GPU (torchrun, one rank per GPU): every rank runs the whole workload on
its own GPU (independent problems, no collective on the data path); the time is
the max over ranks and the value the total work of all ranks over that time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from exact_attention_60_gb300.workloads import WORKLOADS, make_workload_inputs  # noqa: E402

METRIC = "attention fwd TFLOP/s at 1 GB300 and % of dense BF16 tensor peak"
METRIC_BWD = "attention bwd TFLOP/s at 1 GB300 and % of dense BF16 tensor peak"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "seq16k_d128_causal"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
KERNEL_NAME = "fa_fwd_kernel"


# ----------------------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                data = json.load(f)
            return data, "measured"
        except (OSError, ValueError):
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def peak_value(peaks: dict, key: str, default: float) -> float:
    v = peaks.get(key)
    if isinstance(v, dict):  # tolerate {"value": x, ...}
        v = v.get("value")
    try:
        return float(v)
    except (TypeError, ValueError):
        return default


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.error = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError as e:
            self.error = str(e)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"error": self.error or "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"error": "no clock samples"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 or n_gpus > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=os.environ.get("BENCH_DIST_BACKEND", "nccl"))
        return dist, dist.get_rank(), dist.get_world_size(), local
    return None, rank, world, local


def reduce_max(dist, value: float, device=None) -> float:
    """Max of a float over all ranks (a timing reduction, not part of the data path)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(world: int, flops_per_step: float, steps: int, max_ms: float) -> float:
    """Whole-job throughput: every rank ran `steps` steps of `flops_per_step` work;
    the job took the slowest rank's time."""
    return world * flops_per_step * steps / (max_ms / 1e3) / 1e12


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in ("exact_attention_60_gb300/csrc/fa_fwd.cu", "exact_attention_60_gb300/csrc/sm103_ptx.cuh"):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu capture, or None when the
    capture was taken on a different kernel source (or never for this workload)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        data = json.load(f)
    if data.get("kernel_source_sha256") != kernel_source_hash():
        return None
    entry = data.get("workloads", {}).get(workload)
    return None if entry is None else entry["bytes_per_launch"]


# ----------------------------------------------------------------------------- CPU oracle legs
def row_flops(w, rows) -> int:
    """4 D flops per allowed (row, key) pair of the sampled rows."""
    total = 0
    for i in rows:
        lo, hi = w.key_range(int(i))
        total += hi - lo + 1
    return 4 * w.D * total


def time_oracle(w, q, k, v, budget_s: float, heads: int = 2, rows_per_call: int = 64, seed: int = 0):
    """Run the oracle on batches of sampled rows of a few heads until ``budget_s``
    seconds of oracle time are spent; return (flops, seconds, rows, threads)."""
    import oracle
    rng = np.random.default_rng(seed)
    head_ids = rng.choice(w.B * w.H, size=min(heads, w.B * w.H), replace=False)
    per_head = []
    for bh in head_ids:
        b, h = divmod(int(bh), w.H)
        per_head.append(tuple(np.ascontiguousarray(t[b, h].float().numpy(), dtype=np.float64)
                              for t in (q, k, v)))
    flops = 0
    spent = 0.0
    nrows = 0
    it = 0
    while spent < budget_s:
        qq, kk, vv = per_head[it % len(per_head)]
        rows = rng.integers(0, w.Lq, size=rows_per_call)
        t0 = time.perf_counter()
        if w.window is not None:
            oracle.attn_head_window(qq, kk, vv, w.window[0], w.window[1], w.scale, rows=rows)
        else:
            oracle.attn_head(qq, kk, vv, w.causal, w.scale, rows=rows)
        spent += time.perf_counter() - t0
        flops += row_flops(w, rows)
        nrows += rows_per_call
        it += 1
    return flops, spent, nrows, oracle.max_threads()


# ----------------------------------------------------------------------------- arms
def run_reference(args, w):
    """The fp64 CPU oracle as the measured arm: each step is a bounded row sample."""
    dist, rank, world, _ = dist_setup(args.gpus)
    if rank != 0:
        return 0
    q, k, v = make_workload_inputs(w)
    per_step = max(0.5, min(args.ref_seconds_per_step, 120.0 / args.steps))
    for s in range(args.warmup):
        time_oracle(w, q, k, v, per_step / 4, seed=1000 + s)
    tot_flops = 0
    tot_time = 0.0
    tot_rows = 0
    threads = 1
    for s in range(args.steps):
        f, t, n, threads = time_oracle(w, q, k, v, per_step, seed=s)
        tot_flops += f
        tot_time += t
        tot_rows += n
    value = tot_flops / tot_time / 1e12
    sample = (f"{tot_rows} query rows sampled uniformly from 2 heads of the workload, "
              f"about {per_step:g} s of oracle time per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * tot_time / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "shape": w.describe()},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, w):
    import torch
    import exact_attention_60_gb300 as fa
    from exact_attention_60_gb300 import build as fa_build

    fa_build.build()   # no-op when the library is up to date
    fa._native.load()
    dist, rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)

    q_h, k_h, v_h = make_workload_inputs(w)
    # Variants of the same workload (fa_fwd_strided): fp16 values, Q/K/V read in place
    # from [B, L, H, D] memory, per-batch key padding.
    variant = args.dtype != "bf16" or args.layout != "bhld" or args.kv_pad > 0
    io_dtype = torch.float16 if args.dtype == "fp16" else torch.bfloat16
    if args.dtype == "fp16":
        q_h, k_h, v_h = (t.to(torch.float16) for t in (q_h, k_h, v_h))
    kv_len_h = None
    if args.kv_pad > 0:
        g = np.random.default_rng(0xCAFE + w.index)
        lo = max(1, int(round(w.Lk * (1.0 - 2.0 * args.kv_pad))))
        kv_len_h = g.integers(lo, w.Lk + 1, size=w.B).astype(np.int32)
    in_bytes = sum(t.numel() * t.element_size() for t in (q_h, k_h, v_h))
    out_bytes = q_h.numel() * 2 + w.B * w.H * w.Lq * 4
    n_copies = max(2, math.ceil(2 * L2_BYTES / (in_bytes + out_bytes)) + 1)
    bufs = []

    def place(t):   # [B, H, L, D] values, stored [B, L, H, D] with --layout bshd
        t = t.to(dev)
        return t.transpose(1, 2).contiguous().transpose(1, 2) if args.layout == "bshd" else t

    base = tuple(place(t) for t in (q_h, k_h, v_h))
    for c in range(n_copies):
        qkv = base if c == 0 else tuple(place(t) for t in (q_h, k_h, v_h))
        o = torch.empty((w.B, w.H, w.Lq, w.D), device=dev, dtype=io_dtype)
        lse = torch.empty((w.B, w.H, w.Lq), device=dev, dtype=torch.float32)
        bufs.append((*qkv, o, lse))
    kv_len = torch.from_numpy(kv_len_h).to(dev) if kv_len_h is not None else None
    torch.cuda.synchronize(dev)

    # Workspace for the split-key schedule, allocated once outside the timed region
    # (zero bytes, and plain fa_fwd semantics, for causal workloads).
    # Local-window workloads run fa_fwd_window (whole units, no workspace).
    if w.window is None and kv_len is None:
        st, ws_bytes = fa.fa_fwd_workspace_size(w.B, w.H, w.Lq, w.Lk, w.D, w.causal)
        if st != fa.FA_OK:
            raise RuntimeError(fa.fa_status_string(st))
    else:
        ws_bytes = 0
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None
    left, right = w.window if w.window is not None else (-1, 0 if w.causal else -1)
    code = fa.FA_DTYPE_FP16 if args.dtype == "fp16" else fa.FA_DTYPE_BF16

    def launch(i):
        q, k, v, o, lse = bufs[i % n_copies]
        if variant:
            st = fa.fa_fwd_strided(q, q.stride()[:3], k, k.stride()[:3], v, v.stride()[:3], o,
                                   o.stride()[:3], lse, kv_len, w.B, w.H, w.Lq, w.Lk, w.D, left,
                                   right, w.scale, code, ws, ws_bytes, stream)
        elif w.window is not None:
            st = fa.fa_fwd_window(q, k, v, o, lse, w.B, w.H, w.Lq, w.Lk, w.D, w.window[0],
                                  w.window[1], w.scale, stream)
        else:
            st = fa.fa_fwd_ws(q, k, v, o, lse, w.B, w.H, w.Lq, w.Lk, w.D, w.causal, w.scale, ws,
                              ws_bytes, stream)
        if st != fa.FA_OK:
            raise RuntimeError(fa.fa_status_string(st))

    for i in range(args.warmup):
        launch(i)
    torch.cuda.synchronize(dev)
    st = fa.fa_last_device_status(stream)
    if st != fa.FA_OK:
        raise RuntimeError(f"warm-up reported {fa.fa_status_string(st)}")

    sampler = ClockSampler(local)
    if not args.no_clocks:
        sampler.start()
        time.sleep(0.3)
    # ---------------- timed region: K launches, CUDA events on the launching stream
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    # One event pair around the K back-to-back launches (events between them would keep
    # consecutive launches from overlapping their set-up, as a caller's loop does); the
    # attention kernel is the only kernel in the stream, so its mean launch duration is
    # total / K (a split step's combine kernel included).
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record(stream)
    for i in range(args.steps):
        launch(i)
    ev[1].record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    clocks = sampler.stop() if not args.no_clocks else None
    total_ms = ev[0].elapsed_time(ev[1])
    per_launch_ms = [total_ms / args.steps]
    st = fa.fa_last_device_status(stream)
    if st != fa.FA_OK:
        raise RuntimeError(f"timed region reported {fa.fa_status_string(st)}")
    max_ms = reduce_max(dist, total_ms, dev)
    flops = w.flops()
    if kv_len_h is not None:   # only the unpadded pairs count
        i = np.arange(w.Lq, dtype=np.int64)
        lo = np.zeros_like(i) if left < 0 else np.maximum(0, i - left)
        hi_band = np.full_like(i, w.Lk - 1) if right < 0 else np.minimum(w.Lk - 1, i + right)
        pairs = sum(int(np.maximum(0, np.minimum(hi_band, kl - 1) - lo + 1).sum()) for kl in kv_len_h)
        flops = 4 * w.D * w.H * pairs
    value = aggregate_tflops(world, flops, args.steps, max_ms)
    ms_per_step = max_ms / args.steps
    kernel_tflops = flops / (statistics.mean(per_launch_ms) / 1e3) / 1e12

    # ---------------- end to end: pinned host buffers through the public call
    e2e = None
    if not args.skip_e2e and not variant:
        q_p, k_p, v_p = (t.pin_memory() for t in (q_h, k_h, v_h))
        o_p = torch.empty(q_h.shape, dtype=torch.bfloat16).pin_memory()
        l_p = torch.empty((w.B, w.H, w.Lq), dtype=torch.float32).pin_memory()

        def e2e_step():
            # the public host-buffer call: uploads, kernels and downloads overlapped by chunk
            fa.attention_from_host(q_p, k_p, v_p, causal=w.causal, scale=w.scale, out=o_p,
                                   lse=l_p, device=dev, window=w.window)

        e2e_steps = max(1, min(args.steps, 10))
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        barrier(dist, dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = reduce_max(dist, e0.elapsed_time(e1), dev)
        e2e = {"value": aggregate_tflops(world, flops, e2e_steps, e2e_ms), "unit": UNIT,
               "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes,
               "ms_per_step": e2e_ms / e2e_steps}

    peaks, peak_src = load_peaks()
    peak = peak_value(peaks, "bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    hbm_peak = peak_value(peaks, "hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    traffic = measured_traffic(w.name) if not variant else None   # measured on bf16, [B,H,L,D]
    # The bound is the roof the workload's algorithmic intensity (flops per algorithmic
    # byte: Q, K, V read once, O and LSE written once) meets first; both are reported.
    alg_bytes = w.algorithmic_bytes()
    if kv_len_h is not None:   # padded keys are never read
        kv_bytes = 2 * 2 * w.H * w.D * int(kv_len_h.sum())
        alg_bytes = alg_bytes - 2 * 2 * w.B * w.H * w.Lk * w.D + kv_bytes
    launch_s = statistics.mean(per_launch_ms) / 1e3
    hbm_gbs = alg_bytes / launch_s / 1e9
    tensor_bound = flops / alg_bytes >= peak * 1e12 / (hbm_peak * 1e9)
    if tensor_bound:
        roofline = {"bound": "tensor", "achieved": kernel_tflops, "peak": peak, "unit": UNIT,
                    "frac": kernel_tflops / peak, "peak_source": f"{peak_src} bf16 dense (burst)"}
    else:
        roofline = {"bound": "hbm", "achieved": hbm_gbs, "peak": hbm_peak, "unit": "GB/s",
                    "frac": hbm_gbs / hbm_peak, "peak_source": f"{peak_src} HBM copy"}
    roofline.update({"traffic": traffic, "kernel": f"{KERNEL_NAME}<{w.D}>",
                     "algorithmic_bytes": alg_bytes, "flops_per_byte": flops / alg_bytes,
                     "tensor_frac": kernel_tflops / peak, "hbm_achieved_gbs": hbm_gbs,
                     "hbm_frac": hbm_gbs / hbm_peak})

    cpu = None
    if rank == 0 and not args.skip_cpu_baseline:
        f, t, n, threads = time_oracle(w, q_h, k_h, v_h, args.cpu_seconds)
        cpu = {"value": f / t / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{n} query rows sampled uniformly from 2 heads of {w.name}, "
                         f"{t:.1f} s of fp64 oracle time"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": args.dtype,
            "data": "synthetic",
            "config": {"workload": w.name, "shape": w.describe(),
                       "flops_per_step": flops, "io_dtype": args.dtype, "layout": args.layout,
                       "kv_len": None if kv_len_h is None else [int(x) for x in kv_len_h],
                       "l2": f"inputs rotate over {n_copies} copies "
                             f"({n_copies * (in_bytes + out_bytes) / 2**20:.0f} MiB > 2x L2)",
                       "parallelism": f"replica per GPU x{world}",
                       "schedule": ("local-window band" if w.window is not None else
                                    "split key ranges" if ws_bytes else "whole units"),
                       "workspace_bytes": ws_bytes},
            "pct_of_peak": 100.0 * kernel_tflops / peak,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "gpu_launches": args.steps,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def time_oracle_bwd(w, q, k, v, budget_s: float):
    """The oracle's backward on one head of the workload cut to at most 1024 query and key
    rows, repeated until ``budget_s`` seconds: (flops, seconds, calls, threads)."""
    import oracle
    L = min(w.Lq, w.Lk, 1024)
    qq, kk, vv = (np.ascontiguousarray(t[0, 0, :L].float().numpy(), dtype=np.float64) for t in (q, k, v))
    g = np.random.default_rng(0).standard_normal(qq.shape)
    left, right = w.window if w.window is not None else (-1, 0 if w.causal else -1)
    i = np.arange(L)
    lo = np.zeros_like(i) if left < 0 else np.maximum(0, i - left)
    hi = np.full_like(i, L - 1) if right < 0 else np.minimum(L - 1, i + right)
    flops = 2.5 * 4 * w.D * int((hi - lo + 1).sum())
    spent, calls = 0.0, 0
    while spent < budget_s or calls == 0:
        t0 = time.perf_counter()
        oracle.attn_bwd_head_masked(qq, kk, vv, g, left, right, L, w.scale)
        spent += time.perf_counter() - t0
        calls += 1
    return flops * calls, spent, calls, oracle.max_threads(), L


def run_backward(args, w):
    """One step = one fa_bwd call (Delta, dK/dV and dQ kernels) on resident inputs; the
    forward outputs it needs are computed once, outside the timed region."""
    import torch
    import exact_attention_60_gb300 as fa
    from exact_attention_60_gb300 import build as fa_build

    fa_build.build()
    fa._native.load()
    dist, rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    io_dtype = torch.float16 if args.dtype == "fp16" else torch.bfloat16
    variant = args.dtype != "bf16" or args.layout != "bhld" or args.kv_pad > 0 or w.window is not None
    q_h, k_h, v_h = (t.to(io_dtype) for t in make_workload_inputs(w))
    g = torch.Generator().manual_seed(w.seed + 99)
    do_h = torch.randn(q_h.shape, generator=g).to(io_dtype)
    kv_len_h = None
    if args.kv_pad > 0:
        rng = np.random.default_rng(0xCAFE + w.index)
        lo_k = max(1, int(round(w.Lk * (1.0 - 2.0 * args.kv_pad))))
        kv_len_h = rng.integers(lo_k, w.Lk + 1, size=w.B).astype(np.int32)
    kv_len = torch.from_numpy(kv_len_h).to(dev) if kv_len_h is not None else None
    left, right = w.window if w.window is not None else (-1, 0 if w.causal else -1)

    def place(t):   # [B, H, L, D] values, stored [B, L, H, D] with --layout bshd
        t = t.to(dev)
        return t.transpose(1, 2).contiguous().transpose(1, 2) if args.layout == "bshd" else t

    per_copy = 2 * (3 * q_h.numel() + 4 * k_h.numel()) + 8 * w.B * w.H * w.Lq
    n_copies = max(2, math.ceil(2 * L2_BYTES / per_copy) + 1)
    bufs = []
    for c in range(n_copies):
        q, k, v, do = (place(t) for t in (q_h, k_h, v_h, do_h))
        o, lse = fa.attention(q, k, v, causal=w.causal, scale=w.scale, window=w.window, kv_len=kv_len)
        grads = tuple(place(torch.empty(t.shape, dtype=io_dtype)) for t in (q_h, k_h, v_h))
        bufs.append((q, k, v, o, do, lse, *grads))
    st, ws_bytes = fa.fa_bwd_workspace_size(w.B, w.H, w.Lq, w.Lk, w.D, w.causal)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize(dev)
    code = fa.FA_DTYPE_FP16 if args.dtype == "fp16" else fa.FA_DTYPE_BF16

    def launch(i):
        q, k, v, o, do, lse, dq, dk, dv = bufs[i % n_copies]
        if variant:
            st = fa.fa_bwd_strided(q, q.stride()[:3], k, k.stride()[:3], v, v.stride()[:3], o,
                                   o.stride()[:3], do, do.stride()[:3], lse, dq, dq.stride()[:3], dk,
                                   dk.stride()[:3], dv, dv.stride()[:3], kv_len, w.B, w.H, w.Lq, w.Lk,
                                   w.D, left, right, w.scale, code, ws, ws_bytes, stream)
        else:
            st = fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, w.B, w.H, w.Lq, w.Lk, w.D, w.causal,
                           w.scale, ws, ws_bytes, stream)
        if st != fa.FA_OK:
            raise RuntimeError(fa.fa_status_string(st))

    for i in range(args.warmup):
        launch(i)
    torch.cuda.synchronize(dev)
    if fa.fa_last_device_status(stream) != fa.FA_OK:
        raise RuntimeError("warm-up reported a device error")
    sampler = ClockSampler(local)
    if not args.no_clocks:
        sampler.start()
        time.sleep(0.3)
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record(stream)
    for i in range(args.steps):
        launch(i)
    ev[1].record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    clocks = sampler.stop() if not args.no_clocks else None
    if fa.fa_last_device_status(stream) != fa.FA_OK:
        raise RuntimeError("timed region reported a device error")
    max_ms = reduce_max(dist, ev[0].elapsed_time(ev[1]), dev)
    pairs_flops = w.flops()
    if kv_len_h is not None:   # only the unpadded pairs count
        i = np.arange(w.Lq, dtype=np.int64)
        lo = np.zeros_like(i) if left < 0 else np.maximum(0, i - left)
        hi_band = np.full_like(i, w.Lk - 1) if right < 0 else np.minimum(w.Lk - 1, i + right)
        pairs = sum(int(np.maximum(0, np.minimum(hi_band, kl - 1) - lo + 1).sum()) for kl in kv_len_h)
        pairs_flops = 4 * w.D * w.H * pairs
    flops = 2.5 * pairs_flops   # five GEMMs of the forward's size (dV, dP, dS K, dS^T Q, and S)
    value = aggregate_tflops(world, flops, args.steps, max_ms)
    per_gpu = flops / (max_ms / args.steps / 1e3) / 1e12
    peaks, peak_src = load_peaks()
    peak = peak_value(peaks, "bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    cpu = None
    if rank == 0 and not args.skip_cpu_baseline:
        f, t, n, threads, L = time_oracle_bwd(w, q_h, k_h, v_h, args.cpu_seconds)
        cpu = {"value": f / t / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{n} backward passes of head 0 cut to {L} query and key rows, "
                         f"{t:.1f} s of fp64 oracle time"}
    if rank == 0:
        line = {
            "metric": METRIC_BWD, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": max_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": args.dtype,
            "data": "synthetic",
            "config": {"workload": w.name, "shape": w.describe(), "pass": "backward",
                       "io_dtype": args.dtype, "layout": args.layout,
                       "kv_len": None if kv_len_h is None else [int(x) for x in kv_len_h],
                       "flops_per_step": flops, "flop_count": "2.5x forward (five GEMMs); the "
                       "kernels execute seven (dQ is computed apart from dK, dV)",
                       "l2": f"inputs rotate over {n_copies} copies (> 2x L2)",
                       "parallelism": f"replica per GPU x{world}", "workspace_bytes": ws_bytes},
            "pct_of_peak": 100.0 * per_gpu / peak,
            "roofline": {"bound": "tensor", "achieved": per_gpu, "peak": peak, "unit": UNIT,
                         "frac": per_gpu / peak, "traffic": None,
                         "peak_source": f"{peak_src} bf16 dense (burst)",
                         "kernel": f"fa_bwd (Delta + fa_bwd_dkdv_kernel<{w.D}> + fa_bwd_dq_kernel<{w.D}>), "
                                   "whole pass"},
            "cpu_baseline": cpu, "e2e": None, "clocks": clocks, "gpu_launches": 3 * args.steps,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds-per-step", type=float, default=5.0)
    ap.add_argument("--pass", dest="which", choices=["forward", "backward"], default="forward",
                    help="forward (the headline metric) or backward (fa_bwd)")
    ap.add_argument("--dtype", choices=["bf16", "fp16"], default="bf16",
                    help="forward I/O type (fp16 runs fa_fwd_strided)")
    ap.add_argument("--layout", choices=["bhld", "bshd"], default="bhld",
                    help="bshd: Q, K, V stored [B, L, H, D] and read in place (fa_fwd_strided)")
    ap.add_argument("--kv-pad", type=float, default=0.0,
                    help="mean fraction of padded keys per batch (key-padding mask, fa_fwd_strided)")
    args = ap.parse_args(argv)
    if args.warmup < 0 or args.steps < 1:
        ap.error("need --steps >= 1 and --warmup >= 0")
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    if args.which == "backward":
        return run_backward(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
