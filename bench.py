"""Benchmark: attention forward TFLOP/s on one GB300 (and % of dense bf16 peak).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--pass forward|backward]

One step = one fa_fwd launch over the whole workload (every batch, head and
query tile), inputs already resident in HBM.  TFLOP/s counts 4*D flops per
unmasked (query, key) pair.  Between timed steps the inputs rotate over enough
copies that their total exceeds twice the L2 cache.

Prints ONE JSON line (rank 0).  Besides the device-timed value it reports:
  e2e          the same metric through the C host-buffer call fa_fwd_host (pinned
               host Q, K, V in, host O, LSE out; the library overlaps the copies and
               kernels by chunks of heads) with every copy inside the timed region,
               beside the time one plain upload of the inputs takes;
  roofline     achieved TFLOP/s of the kernel against the measured bf16 peak (or GB/s
               against the measured copy rate, whichever roof the workload meets first);
  cpu_baseline the fp64 oracle timed on the host cores on a bounded row sample;
  clocks       SM clocks, power and throttle reasons sampled during the timed region;
  per_config   every configuration of the specification (C1-C5, C2 with both masks),
               the two local-attention workloads and the 16K causal backward pass,
               each timed over at least --per-config-seconds of back-to-back launches
               with its own roofline and the clock samples taken inside that window.
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


class NvmlReader:
    """Read-only NVML queries through ctypes: SM clock, its maximum, board power and the
    active clock-event (throttle) reasons of one GPU, found by PCI bus id.  NVML ships
    with the driver; `lib` may be a stand-in object with the same functions (tests)."""
    CLOCK_SM = 1
    # Public NVML clock-event reason bits.
    REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40}

    def __init__(self, pci_bus_id: str, lib=None):
        import ctypes
        self.ct = ctypes
        self.lib = lib if lib is not None else ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.handle = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(),
                                                     ctypes.byref(self.handle)) != 0:
            self.lib.nvmlShutdown()
            raise OSError(f"no NVML device at {pci_bus_id}")
        self.reasons_fn = (getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or
                           getattr(self.lib, "nvmlDeviceGetCurrentClocksThrottleReasons", None))
        v = ctypes.c_uint()
        self.max_mhz = (float(v.value) if self.lib.nvmlDeviceGetMaxClockInfo(
            self.handle, self.CLOCK_SM, ctypes.byref(v)) == 0 else None)

    def sample(self, with_power: bool):
        """(sm MHz, max MHz, power W or None, set of reason names), or None on an error."""
        ct = self.ct
        v = ct.c_uint()
        if self.lib.nvmlDeviceGetClockInfo(self.handle, self.CLOCK_SM, ct.byref(v)) != 0:
            return None
        sm = float(v.value)
        power = None
        if with_power and self.lib.nvmlDeviceGetPowerUsage(self.handle, ct.byref(v)) == 0:
            power = v.value / 1000.0
        reasons = set()
        if self.reasons_fn is not None:
            r = ct.c_ulonglong()
            if self.reasons_fn(self.handle, ct.byref(r)) == 0:
                reasons = {n for n, bit in self.REASON_BITS.items() if r.value & bit}
        return sm, (self.max_mhz if self.max_mhz is not None else sm), power, reasons

    def close(self):
        self.lib.nvmlShutdown()


def pci_bus_id_of(index: int):
    """NVML-style PCI bus id (domain:bus:device.function) of CUDA device `index`."""
    import torch
    p = torch.cuda.get_device_properties(index)
    try:
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except AttributeError:
        return None


class ClockSampler:
    """SM clocks, power and throttle reasons sampled while running.

    Preferred source: NVML, polled from a thread every `period_ms` (2 ms by default, so
    that a timed region of a few milliseconds still holds samples).  Fallback: nvidia-smi
    at its 100 ms loop.  Every sample carries a host timestamp (time.time()), so
    ``summary(t0, t1)`` can keep only the samples taken inside a timed window."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int, period_ms: float = 2.0, nvml=None):
        self.gpu_index = gpu_index
        self.period_ms = period_ms
        self.nvml = nvml          # an NvmlReader, made in start() when not given
        self.proc = None
        self.thread = None
        self.lines = []           # nvidia-smi CSV lines (fallback)
        self.polled = []          # NVML samples (t, sm, smax, power, reasons)
        self.source = None
        self.error = None
        self._stop = threading.Event()

    def start(self):
        if self.nvml is None:
            try:
                bus = pci_bus_id_of(self.gpu_index)
                if bus is not None:
                    self.nvml = NvmlReader(bus)
            except (OSError, AttributeError, RuntimeError) as e:
                self.error = f"NVML: {e}"
                self.nvml = None
        if self.nvml is not None:
            self.source = f"NVML every {self.period_ms:g} ms"
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi every 100 ms"
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError as e:
            self.error = str(e)

    def _poll(self):
        n = 0
        while not self._stop.is_set():
            # Board power is the slowest query: every other sample only.
            x = self.nvml.sample(with_power=(n % 2 == 0))
            if x is not None:
                self.polled.append((time.time(),) + x)
            n += 1
            self._stop.wait(self.period_ms / 1000.0)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def _samples(self):
        import datetime
        out = list(self.polled)
        for line in list(self.lines):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                t = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm, smax = float(parts[2]), float(parts[3])
            except ValueError:
                continue
            try:
                power = float(parts[4])
            except ValueError:
                power = None
            reasons = {n for n, v in zip(self.REASONS, parts[6:10]) if v.lower() == "active"}
            out.append((t, sm, smax, power, reasons))
        return out

    def summary(self, t0=None, t1=None):
        """Median SM clock, max clock, throttle reasons and power over the samples taken in
        [t0, t1] (all samples when no window is given or none falls inside it)."""
        samples = self._samples()
        if not samples:
            return {"error": self.error or "no clock samples"}
        inside = [x for x in samples if t0 is not None and t0 <= x[0] <= t1]
        use = inside if inside else samples
        power = [x[3] for x in use if x[3] is not None]
        res = {"sm_mhz": statistics.median(x[1] for x in use),
               "sm_max_mhz": max(x[2] for x in use),
               "reasons": sorted(set().union(*(x[4] for x in use))),
               "samples": len(use), "samples_in_window": len(inside),
               "power_w_max": max(power) if power else None}
        if t0 is not None:
            res["window_s"] = t1 - t0
        if self.source:
            res["source"] = self.source
        return res

    def stop(self):
        self._stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)
        if self.nvml is not None:
            try:
                self.nvml.close()
            except OSError:
                pass


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
    # Every host core this process may run on, whatever OMP_NUM_THREADS says (a multi-process
    # launcher sets it to 1 for each rank, and only one rank times the oracle).
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    flops = 0
    spent = 0.0
    nrows = 0
    it = 0
    while spent < budget_s:
        qq, kk, vv = per_head[it % len(per_head)]
        rows = rng.integers(0, w.Lq, size=rows_per_call)
        t0 = time.perf_counter()
        if w.window is not None:
            oracle.attn_head_window(qq, kk, vv, w.window[0], w.window[1], w.scale, rows=rows,
                                    nthreads=threads)
        else:
            oracle.attn_head(qq, kk, vv, w.causal, w.scale, rows=rows, nthreads=threads)
        spent += time.perf_counter() - t0
        flops += row_flops(w, rows)
        nrows += rows_per_call
        it += 1
    return flops, spent, nrows, threads


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


class ForwardSetup:
    """Device buffers of one forward workload, rotated over enough copies that their
    total exceeds twice the L2 cache, and ``launch(i)`` for step i (a public C call)."""

    def __init__(self, fa, w, dev, stream, dtype="bf16", layout="bhld", kv_pad=0.0):
        import torch
        self.fa, self.w, self.dev, self.stream = fa, w, dev, stream
        q_h, k_h, v_h = make_workload_inputs(w)
        # Variants of the same workload (fa_fwd_strided): fp16 values, Q/K/V read in place
        # from [B, L, H, D] memory, per-batch key padding.
        self.variant = dtype != "bf16" or layout != "bhld" or kv_pad > 0
        io_dtype = torch.float16 if dtype == "fp16" else torch.bfloat16
        if dtype == "fp16":
            q_h, k_h, v_h = (t.to(torch.float16) for t in (q_h, k_h, v_h))
        self.host = (q_h, k_h, v_h)
        self.kv_len_h = None
        if kv_pad > 0:
            g = np.random.default_rng(0xCAFE + w.index)
            lo = max(1, int(round(w.Lk * (1.0 - 2.0 * kv_pad))))
            self.kv_len_h = g.integers(lo, w.Lk + 1, size=w.B).astype(np.int32)
        self.in_bytes = sum(t.numel() * t.element_size() for t in (q_h, k_h, v_h))
        self.out_bytes = q_h.numel() * 2 + w.B * w.H * w.Lq * 4
        self.n_copies = max(2, math.ceil(2 * L2_BYTES / (self.in_bytes + self.out_bytes)) + 1)

        def place(t):   # [B, H, L, D] values, stored [B, L, H, D] with layout bshd
            t = t.to(dev)
            return t.transpose(1, 2).contiguous().transpose(1, 2) if layout == "bshd" else t

        base = tuple(place(t) for t in (q_h, k_h, v_h))
        self.bufs = []
        for c in range(self.n_copies):
            qkv = base if c == 0 else tuple(place(t) for t in (q_h, k_h, v_h))
            o = torch.empty((w.B, w.H, w.Lq, w.D), device=dev, dtype=io_dtype)
            lse = torch.empty((w.B, w.H, w.Lq), device=dev, dtype=torch.float32)
            self.bufs.append((*qkv, o, lse))
        self.kv_len = torch.from_numpy(self.kv_len_h).to(dev) if self.kv_len_h is not None else None
        # Workspace for the split-key schedule, allocated once outside the timed region
        # (zero bytes, and plain fa_fwd semantics, for causal workloads).  Local-window
        # workloads run fa_fwd_window (whole units, no workspace).
        if w.window is None and self.kv_len is None:
            st, self.ws_bytes = fa.fa_fwd_workspace_size(w.B, w.H, w.Lq, w.Lk, w.D, w.causal)
            if st != fa.FA_OK:
                raise RuntimeError(fa.fa_status_string(st))
        else:
            self.ws_bytes = 0
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev) if self.ws_bytes else None
        # The schedule the library takes (its own answer, not a guess from the sizes).
        if w.window is not None:
            self.schedule = "local-window band"
        elif self.kv_len is not None:
            self.schedule = "band (key padding)"
        else:
            st, sc = fa.fa_fwd_schedule(w.B, w.H, w.Lq, w.Lk, w.D, w.causal)
            if st != fa.FA_OK:
                raise RuntimeError(fa.fa_status_string(st))
            self.schedule = {fa.FA_SCHED_WHOLE: "whole units",
                             fa.FA_SCHED_SPLIT: "split key ranges",
                             fa.FA_SCHED_TABLE: "whole units in host-computed table order"}[sc]
        self.left, self.right = w.window if w.window is not None else (-1, 0 if w.causal else -1)
        self.code = fa.FA_DTYPE_FP16 if dtype == "fp16" else fa.FA_DTYPE_BF16
        torch.cuda.synchronize(dev)

    def launch(self, i):
        fa, w = self.fa, self.w
        q, k, v, o, lse = self.bufs[i % self.n_copies]
        if self.variant:
            st = fa.fa_fwd_strided(q, q.stride()[:3], k, k.stride()[:3], v, v.stride()[:3], o,
                                   o.stride()[:3], lse, self.kv_len, w.B, w.H, w.Lq, w.Lk, w.D,
                                   self.left, self.right, w.scale, self.code, self.ws,
                                   self.ws_bytes, self.stream)
        elif w.window is not None:
            st = fa.fa_fwd_window(q, k, v, o, lse, w.B, w.H, w.Lq, w.Lk, w.D, w.window[0],
                                  w.window[1], w.scale, self.stream)
        else:
            st = fa.fa_fwd_ws(q, k, v, o, lse, w.B, w.H, w.Lq, w.Lk, w.D, w.causal, w.scale,
                              self.ws, self.ws_bytes, self.stream)
        if st != fa.FA_OK:
            raise RuntimeError(fa.fa_status_string(st))

    def flops(self):
        w = self.w
        if self.kv_len_h is None:
            return w.flops()
        i = np.arange(w.Lq, dtype=np.int64)   # only the unpadded pairs count
        lo = np.zeros_like(i) if self.left < 0 else np.maximum(0, i - self.left)
        hi_band = np.full_like(i, w.Lk - 1) if self.right < 0 else np.minimum(w.Lk - 1, i + self.right)
        pairs = sum(int(np.maximum(0, np.minimum(hi_band, kl - 1) - lo + 1).sum()) for kl in self.kv_len_h)
        return 4 * w.D * w.H * pairs

    def algorithmic_bytes(self):
        w = self.w
        alg = w.algorithmic_bytes()
        if self.kv_len_h is not None:   # padded keys are never read
            alg = alg - 2 * 2 * w.B * w.H * w.Lk * w.D + 2 * 2 * w.H * w.D * int(self.kv_len_h.sum())
        return alg

    def free(self):
        import torch
        self.bufs = []
        self.ws = None
        self.kv_len = None
        torch.cuda.empty_cache()


def roofline_of(setup, flops, per_launch_s, peaks, peak_src, traffic, sustained=False):
    """The roof the workload's algorithmic intensity (flops per algorithmic byte: Q, K, V
    read once, O and LSE written once) meets first, and the achieved fraction of it; both
    fractions are reported.  ``sustained``: the kernel ran back to back for a second or
    more, under the power cap, so the sustained bf16 figure is the tensor roof."""
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    peak = peak_value(peaks, key, FALLBACK_PEAKS[key])
    hbm_peak = peak_value(peaks, "hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    alg_bytes = setup.algorithmic_bytes()
    kernel_tflops = flops / per_launch_s / 1e12
    hbm_gbs = alg_bytes / per_launch_s / 1e9
    if flops / alg_bytes >= peak * 1e12 / (hbm_peak * 1e9):
        roof = {"bound": "tensor", "achieved": kernel_tflops, "peak": peak, "unit": UNIT,
                "frac": kernel_tflops / peak,
                "peak_source": f"{peak_src} bf16 dense ({'sustained' if sustained else 'burst'})"}
    else:
        roof = {"bound": "hbm", "achieved": hbm_gbs, "peak": hbm_peak, "unit": "GB/s",
                "frac": hbm_gbs / hbm_peak, "peak_source": f"{peak_src} HBM copy"}
    roof.update({"traffic": traffic, "kernel": f"{KERNEL_NAME}<{setup.w.D}>",
                 "algorithmic_bytes": alg_bytes, "flops_per_byte": flops / alg_bytes,
                 "tensor_frac": kernel_tflops / peak, "hbm_achieved_gbs": hbm_gbs,
                 "hbm_frac": hbm_gbs / hbm_peak})
    return roof


# The specification's configurations, one bench line each in ``per_config``.
PER_CONFIG = [("C1", "tiny_d64"), ("C2", "seq1k_d64"), ("C2-causal", "seq1k_d64_causal"),
              ("C3", "seq4k_d128_causal"), ("C4", "seq16k_d128_causal"),
              ("C5", "cross_q500_k8191_d128")]
# The extensions beyond the forward's plain masks, timed the same way: local attention
# (a causal window and a symmetric band) and the backward pass.
PER_CONFIG_LOCAL = [("window-16k-d128", "seq16k_d128_window4k"), ("local256-4k-d64", "seq4k_d64_local256")]
PER_CONFIG_BACKWARD = [("backward-16k-causal-d128", "seq16k_d128_causal")]


def measure_backward(fa, w, dev, stream, peaks, peak_src, seconds, no_clocks):
    """The backward pass (one fa_bwd call: Delta, dK/dV and dQ kernels) timed over at least
    ``seconds`` of back-to-back calls on resident inputs, clocks sampled inside that window.
    TFLOP/s at the conventional count of five GEMMs of the forward's size."""
    import torch
    q_h, k_h, v_h = make_workload_inputs(w)
    g = torch.Generator().manual_seed(w.seed + 99)
    do_h = torch.randn(q_h.shape, generator=g).to(torch.bfloat16)
    per_copy = 2 * (3 * q_h.numel() + 4 * k_h.numel()) + 8 * w.B * w.H * w.Lq
    n_copies = max(2, math.ceil(2 * L2_BYTES / per_copy) + 1)
    bufs = []
    for c in range(n_copies):
        q, k, v, do = (t.to(dev) for t in (q_h, k_h, v_h, do_h))
        o, lse = fa.attention(q, k, v, causal=w.causal, scale=w.scale)
        bufs.append((q, k, v, o, do, lse, torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)))
    st, ws_bytes = fa.fa_bwd_workspace_size(w.B, w.H, w.Lq, w.Lk, w.D, w.causal)
    if st != fa.FA_OK:
        raise RuntimeError(fa.fa_status_string(st))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

    def launch(i):
        q, k, v, o, do, lse, dq, dk, dv = bufs[i % n_copies]
        st = fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, w.B, w.H, w.Lq, w.Lk, w.D, w.causal,
                       w.scale, ws, ws_bytes, stream)
        if st != fa.FA_OK:
            raise RuntimeError(fa.fa_status_string(st))

    for i in range(3):
        launch(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(5):
        launch(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    est_ms = max(e0.elapsed_time(e1) / 5, 1e-3)
    steps = int(min(100000, max(20, math.ceil(seconds * 1000.0 / est_ms))))
    sampler = ClockSampler(dev.index, period_ms=20.0)
    if not no_clocks:
        sampler.start()
        time.sleep(0.3)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    e0.record(stream)
    for i in range(steps):
        launch(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    if not no_clocks:
        time.sleep(0.15)
        sampler.stop()
    clocks = None if no_clocks else sampler.summary(t0, t1)
    st = fa.fa_last_device_status(stream)
    if st != fa.FA_OK:
        raise RuntimeError(f"{w.name} backward: {fa.fa_status_string(st)}")
    total_ms = e0.elapsed_time(e1)
    flops = 2.5 * w.flops()
    tflops = flops / (total_ms / steps / 1e3) / 1e12
    peak = peak_value(peaks, "bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    entry = {"workload": w.name, "shape": w.describe(), "pass": "backward", "steps": steps,
             "ms_per_step": total_ms / steps, "tflops": tflops,
             "flop_count": "2.5x forward (five GEMMs); the kernels execute seven",
             "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": UNIT,
                          "frac": tflops / peak, "traffic": None,
                          "peak_source": f"{peak_src} bf16 dense (sustained)",
                          "kernel": f"fa_bwd (Delta + fa_bwd_dkdv_kernel<{w.D}> + "
                                    f"fa_bwd_dq_kernel<{w.D}>), whole pass"},
             "clocks": clocks}
    del bufs, ws
    torch.cuda.empty_cache()
    return entry


def measure_config(fa, w, dev, stream, peaks, peak_src, seconds, no_clocks):
    """One configuration timed over at least ``seconds`` of back-to-back launches (one CUDA
    event pair on the launching stream), with the clocks sampled inside that window."""
    import torch
    setup = ForwardSetup(fa, w, dev, stream)
    for i in range(5):
        setup.launch(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(20):
        setup.launch(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    est_ms = max(e0.elapsed_time(e1) / 20, 1e-3)
    steps = int(min(200000, max(50, math.ceil(seconds * 1000.0 / est_ms))))
    # Host cost of one launch (the C call and its argument checks), over fewer launches
    # than the stream's queue holds, so the host never waits for the GPU here.
    torch.cuda.synchronize(dev)
    h0 = time.perf_counter()
    for i in range(100):
        setup.launch(i)
    host_us = (time.perf_counter() - h0) / 100 * 1e6
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(dev.index, period_ms=20.0)
    if not no_clocks:
        sampler.start()
        time.sleep(0.3)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    e0.record(stream)
    for i in range(steps):
        setup.launch(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    if not no_clocks:
        time.sleep(0.15)
        sampler.stop()
    clocks = None if no_clocks else sampler.summary(t0, t1)
    st = fa.fa_last_device_status(stream)
    if st != fa.FA_OK:
        raise RuntimeError(f"{w.name}: {fa.fa_status_string(st)}")
    total_ms = e0.elapsed_time(e1)
    per_launch_s = total_ms / steps / 1e3
    flops = setup.flops()
    entry = {"workload": w.name, "shape": w.describe(), "steps": steps,
             "ms_per_step": total_ms / steps, "tflops": flops / per_launch_s / 1e12,
             "us_per_step": total_ms / steps * 1e3, "host_us_per_launch": host_us,
             "schedule": setup.schedule,
             "roofline": roofline_of(setup, flops, per_launch_s, peaks, peak_src,
                                     measured_traffic(w.name), sustained=True),
             "clocks": clocks}
    if host_us > 0.5 * total_ms / steps * 1e3:
        # The host's launch rate may limit the stream: replay the same launches from a CUDA
        # graph (captured once; no host work per launch) for the device-limited figure.
        entry["graph"] = graph_replay(setup, stream, flops, seconds / 2, est_ms)
    setup.free()
    return entry


def graph_replay(setup, stream, flops, seconds, est_ms):
    import torch
    n = 20
    try:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(setup.dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            setup.stream = side
            with torch.cuda.graph(g, stream=side):
                for i in range(n):
                    setup.launch(i)
    except RuntimeError as e:
        return {"error": str(e)[:200]}
    finally:
        setup.stream = stream
    stream.wait_stream(side)
    reps = int(max(10, math.ceil(seconds * 1000.0 / (n * est_ms))))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize(setup.dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(torch.cuda.current_stream(setup.dev))
    for _ in range(reps):
        g.replay()
    e1.record(torch.cuda.current_stream(setup.dev))
    torch.cuda.synchronize(setup.dev)
    per_step_ms = e0.elapsed_time(e1) / (reps * n)
    return {"steps": reps * n, "us_per_step": per_step_ms * 1e3,
            "tflops": flops / (per_step_ms / 1e3) / 1e12,
            "how": f"{n} launches captured once in a CUDA graph, replayed {reps} times"}


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
    setup = ForwardSetup(fa, w, dev, stream, args.dtype, args.layout, args.kv_pad)
    variant = setup.variant

    for i in range(args.warmup):
        setup.launch(i)
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
    t_begin = time.time()
    ev[0].record(stream)
    for i in range(args.steps):
        setup.launch(i)
    ev[1].record(stream)
    torch.cuda.synchronize(dev)
    t_end = time.time()
    barrier(dist, dev)
    if not args.no_clocks:
        time.sleep(0.15)
        sampler.stop()
    clocks = None if args.no_clocks else sampler.summary(t_begin, t_end)
    total_ms = ev[0].elapsed_time(ev[1])
    st = fa.fa_last_device_status(stream)
    if st != fa.FA_OK:
        raise RuntimeError(f"timed region reported {fa.fa_status_string(st)}")
    max_ms = reduce_max(dist, total_ms, dev)
    flops = setup.flops()
    value = aggregate_tflops(world, flops, args.steps, max_ms)
    ms_per_step = max_ms / args.steps
    per_launch_s = total_ms / args.steps / 1e3
    kernel_tflops = flops / per_launch_s / 1e12
    q_h, k_h, v_h = setup.host
    in_bytes, out_bytes, ws_bytes, n_copies = (setup.in_bytes, setup.out_bytes, setup.ws_bytes,
                                               setup.n_copies)
    kv_len_h = setup.kv_len_h
    schedule = setup.schedule
    peaks, peak_src = load_peaks()
    traffic = measured_traffic(w.name) if not variant else None   # measured on bf16, [B,H,L,D]
    roofline = roofline_of(setup, flops, per_launch_s, peaks, peak_src, traffic)
    peak = roofline["peak"] if roofline["bound"] == "tensor" else peak_value(
        peaks, "bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    setup.free()

    # ---------------- end to end: pinned host buffers through the C call fa_fwd_host
    e2e = None
    if not args.skip_e2e and not variant:
        q_p, k_p, v_p = (t.pin_memory() for t in (q_h, k_h, v_h))
        o_p = torch.empty(q_h.shape, dtype=torch.bfloat16).pin_memory()
        l_p = torch.empty((w.B, w.H, w.Lq), dtype=torch.float32).pin_memory()
        left, right = setup.left, setup.right
        st, host_ws_bytes = fa.fa_fwd_host_workspace_size(w.B, w.H, w.Lq, w.Lk, w.D, left, right)
        if st != fa.FA_OK:
            raise RuntimeError(fa.fa_status_string(st))
        host_ws = torch.empty(max(host_ws_bytes, 256), dtype=torch.uint8, device=dev)   # once

        def e2e_step():
            # uploads, kernels and downloads overlapped by chunks of heads inside the library
            st = fa.fa_fwd_host(q_p, k_p, v_p, o_p, l_p, w.B, w.H, w.Lq, w.Lk, w.D, left, right,
                                w.scale, host_ws, host_ws.numel(), stream)
            if st != fa.FA_OK:
                raise RuntimeError(fa.fa_status_string(st))

        # The host link alone: one upload of the step's inputs, the floor of an e2e step.
        scratch = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
        flat = [t.view(-1).view(torch.uint8) for t in (q_p, k_p, v_p)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        off = 0
        e0.record(stream)
        for t in flat:
            scratch[off:off + t.numel()].copy_(t, non_blocking=True)
            off += t.numel()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        upload_ms = e0.elapsed_time(e1)
        del scratch
        e2e_steps = max(1, min(args.steps, 10))
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        # Three timed windows of e2e_steps calls each; the median window is reported (the
        # host link is shared with the machine's other GPUs, and one window can catch a
        # burst of someone else's copies).  Every window is listed in "windows_ms".
        windows = []
        for _ in range(3):
            barrier(dist, dev)
            e0.record(stream)
            for _ in range(e2e_steps):
                e2e_step()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            if fa.fa_last_device_status(stream) != fa.FA_OK:
                raise RuntimeError("e2e steps reported a device error")
            windows.append(reduce_max(dist, e0.elapsed_time(e1), dev))
        e2e_ms = statistics.median(windows)
        e2e = {"value": aggregate_tflops(world, flops, e2e_steps, e2e_ms), "unit": UNIT,
               "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes,
               "ms_per_step": e2e_ms / e2e_steps, "steps": e2e_steps,
               "windows_ms": [x / e2e_steps for x in windows],
               "call": "fa_fwd_host (C ABI, pinned host buffers, device workspace allocated once)",
               "upload_only_ms": upload_ms, "upload_gbs": in_bytes / upload_ms / 1e6}

    cpu = None
    if rank == 0 and not args.skip_cpu_baseline:
        f, t, n, threads = time_oracle(w, q_h, k_h, v_h, args.cpu_seconds)
        cpu = {"value": f / t / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{n} query rows sampled uniformly from 2 heads of {w.name}, "
                         f"{t:.1f} s of fp64 oracle time"}

    per_config = None
    if rank == 0 and not args.skip_per_config and not variant:
        per_config = {}
        for label, name in PER_CONFIG + PER_CONFIG_LOCAL:
            per_config[label] = measure_config(fa, WORKLOADS[name], dev, stream, peaks, peak_src,
                                               args.per_config_seconds, args.no_clocks)
        for label, name in PER_CONFIG_BACKWARD:
            per_config[label] = measure_backward(fa, WORKLOADS[name], dev, stream, peaks, peak_src,
                                                 args.per_config_seconds, args.no_clocks)

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
                       "schedule": schedule,
                       "workspace_bytes": ws_bytes},
            "pct_of_peak": 100.0 * kernel_tflops / peak,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            # one attention kernel per step; the split-key schedule adds its merge kernel
            "gpu_launches": args.steps * (2 if schedule == "split key ranges" else 1),
            "per_config": per_config,
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
    t_begin = time.time()
    ev[0].record(stream)
    for i in range(args.steps):
        launch(i)
    ev[1].record(stream)
    torch.cuda.synchronize(dev)
    t_end = time.time()
    barrier(dist, dev)
    if not args.no_clocks:
        time.sleep(0.15)
        sampler.stop()
    clocks = None if args.no_clocks else sampler.summary(t_begin, t_end)
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
    ap.add_argument("--skip-per-config", action="store_true",
                    help="skip the per-configuration lines (each timed over >= --per-config-seconds)")
    ap.add_argument("--per-config-seconds", type=float, default=1.0)
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
