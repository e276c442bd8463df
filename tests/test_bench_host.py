"""Host logic of the benchmark: work counts, the DRAM-traffic record and the peak lookup.

The pair counts that every TFLOP/s figure divides by are checked against masks built
element by element from the mask definitions (top-left causal j <= i; band
i - left <= j <= i + right; keys past Lk excluded), and the large workloads against the
closed forms quoted with the measurements.
"""
import json

import numpy as np
import pytest

import bench
from exact_attention_60_gb300.workloads import WORKLOADS, Workload


def brute_pairs(Lq, Lk, causal, window):
    i = np.arange(Lq)[:, None]
    j = np.arange(Lk)[None, :]
    keep = np.ones((Lq, Lk), dtype=bool)
    if window is not None:
        left, right = window
        if left >= 0:
            keep &= j >= i - left
        if right >= 0:
            keep &= j <= i + right
    elif causal:
        keep &= j <= i
    return int(keep.sum())


@pytest.mark.parametrize("Lq,Lk,causal,window", [
    (1, 1, False, None), (1, 1, True, None), (130, 130, True, None), (300, 129, True, None),
    (129, 300, True, None), (500, 257, False, None), (257, 257, False, (100, 0)),
    (257, 257, False, (64, 64)), (257, 400, False, (-1, 3)), (257, 400, False, (200, -1)),
    (257, 257, False, (0, 0)), (64, 500, False, (10, 600)),
])
def test_pairs_per_head_equal_the_mask(Lq, Lk, causal, window):
    w = Workload("t", 1, 1, Lq, Lk, 64, causal, window=window)
    assert w.pairs_per_head() == brute_pairs(Lq, Lk, causal, window)
    # the per-row ranges the CPU baseline's sampled rows use cover the same pairs
    assert sum(hi - lo + 1 for lo, hi in (w.key_range(r) for r in range(Lq))) == w.pairs_per_head()
    assert bench.row_flops(w, range(Lq)) == 4 * w.D * w.pairs_per_head()


def test_workload_flops_closed_forms():
    w = WORKLOADS["seq16k_d128_causal"]
    assert w.flops() == 4 * 128 * 16 * (16384 * 16385 // 2) == 1_099_578_736_640
    w = WORKLOADS["seq4k_d128_causal"]
    assert w.flops() == 4 * 128 * 2 * 32 * (4096 * 4097 // 2)
    w = WORKLOADS["cross_q500_k8191_d128"]
    assert w.flops() == 4 * 128 * 8 * 16 * 500 * 8191
    w = WORKLOADS["seq1k_d64"]
    assert w.flops() == 4 * 64 * 4 * 16 * 1024 * 1024 == 17_179_869_184
    w = WORKLOADS["seq16k_d128_window4k"]   # keys i-4095 .. i
    per_head = sum(min(i, 4095) + 1 for i in range(16384))
    assert w.flops() == 4 * 128 * 16 * per_head


def test_algorithmic_bytes_closed_form():
    # Q, K, V read and O written once in bf16, LSE written once in fp32
    w = WORKLOADS["seq16k_d128_causal"]
    assert w.algorithmic_bytes() == 4 * 16384 * 128 * 2 * 16 + 16 * 16384 * 4 == 269_484_032
    w = WORKLOADS["cross_q500_k8191_d128"]
    bh = 8 * 16
    assert w.algorithmic_bytes() == bh * (2 * 500 + 2 * 8191) * 128 * 2 + bh * 500 * 4


def test_measured_traffic_is_reported_only_for_the_captured_source(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    record = {"kernel_source_sha256": "abc", "workloads": {"seq16k_d128_causal": {"bytes_per_launch": 5.0e8}}}
    (prof / "dram_traffic.json").write_text(json.dumps(record))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "abc")
    assert bench.measured_traffic("seq16k_d128_causal") == 5.0e8
    assert bench.measured_traffic("seq4k_d128_causal") is None       # never captured
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "changed")
    assert bench.measured_traffic("seq16k_d128_causal") is None      # kernel changed since


def test_committed_traffic_record_is_consistent():
    """Each entry's total is its read plus write bytes and its algorithmic bytes are the
    workload's; a record taken on another kernel source is reported by the bench as null."""
    data = json.load(open(bench.os.path.join(bench.ROOT, "profiles", "dram_traffic.json")))
    if data["kernel_source_sha256"] != bench.kernel_source_hash():
        pytest.skip("the traffic record predates the current kernel source (bench reports null)")
    for name, entry in data["workloads"].items():
        assert entry["bytes_per_launch"] == entry["dram_bytes_read"] + entry["dram_bytes_write"]
        assert entry["algorithmic_bytes"] == WORKLOADS[name].algorithmic_bytes()


def test_peak_lookup():
    assert bench.peak_value({"bf16_tflops": 1911.6}, "bf16_tflops", 1.0) == 1911.6
    assert bench.peak_value({"bf16_tflops": {"value": "1800"}}, "bf16_tflops", 1.0) == 1800.0
    assert bench.peak_value({"bf16_tflops": None}, "bf16_tflops", 7.0) == 7.0
    assert bench.peak_value({}, "hbm_gbs", 6800.0) == 6800.0
    peaks, source = bench.load_peaks()
    assert source in ("measured", "fallback")
    assert bench.peak_value(peaks, "bf16_tflops", 0.0) > 0


def test_clock_sampler_keeps_samples_inside_the_window():
    import datetime
    s = bench.ClockSampler(0)
    base = datetime.datetime(2026, 1, 2, 3, 4, 5)
    def line(dt_s, mhz, power, cap):
        t = (base + datetime.timedelta(seconds=dt_s)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return f"{t}, 0, {mhz}, 2070, {power}, 0x0, Not Active, Not Active, Not Active, {cap}"
    s.lines = [line(0.0, 1000, 200.0, "Not Active"), line(0.5, 1900, 1300.0, "Active"),
               line(0.6, 1700, 1350.0, "Active"), line(0.7, 1800, 1390.0, "Not Active"),
               line(2.0, 900, 180.0, "Not Active"), "garbage line"]
    t0 = (base + datetime.timedelta(seconds=0.45)).timestamp()
    t1 = (base + datetime.timedelta(seconds=0.75)).timestamp()
    r = s.summary(t0, t1)
    assert r["samples_in_window"] == 3 and r["samples"] == 3
    assert r["sm_mhz"] == 1800 and r["sm_max_mhz"] == 2070
    assert r["reasons"] == ["sw_power_cap"] and r["power_w_max"] == 1390.0
    # a window with no sample falls back to every sample, and says so
    r = s.summary(t1 + 10, t1 + 11)
    assert r["samples_in_window"] == 0 and r["samples"] == 5
    assert bench.ClockSampler(0).summary()["error"]


class _FakeNvml:
    """Stand-in for the NVML library: a clock that steps through `mhz`, and the
    sw_power_cap reason bit from the third sample on."""
    def __init__(self, mhz):
        self.mhz = list(mhz)
        self.n = 0
        self.closed = False

    def nvmlInit_v2(self):
        return 0

    def nvmlShutdown(self):
        self.closed = True
        return 0

    def nvmlDeviceGetHandleByPciBusId_v2(self, bus, ref):
        assert bus == b"00000000:01:00.0"
        ref._obj.value = 1234
        return 0

    def nvmlDeviceGetMaxClockInfo(self, h, clock, ref):
        assert clock == 1
        ref._obj.value = 2070
        return 0

    def nvmlDeviceGetClockInfo(self, h, clock, ref):
        ref._obj.value = self.mhz[min(self.n, len(self.mhz) - 1)]
        self.n += 1
        return 0

    def nvmlDeviceGetPowerUsage(self, h, ref):
        ref._obj.value = 1380000   # milliwatts
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, h, ref):
        ref._obj.value = 0x4 | 0x1 if self.n >= 3 else 0x1   # sw_power_cap (+ idle bit)
        return 0


def test_nvml_sampler_reads_clocks_power_and_reasons_from_a_fake_library():
    import time as _time
    lib = _FakeNvml([2070, 2070, 1800, 1700, 1700])
    reader = bench.NvmlReader("00000000:01:00.0", lib=lib)
    assert reader.max_mhz == 2070.0
    sm, smax, power, reasons = reader.sample(with_power=True)
    assert (sm, smax, power, reasons) == (2070.0, 2070.0, 1380.0, set())
    s = bench.ClockSampler(0, period_ms=1.0, nvml=reader)
    t0 = _time.time()
    s.start()
    _time.sleep(0.05)
    s.stop()
    t1 = _time.time()
    r = s.summary(t0, t1)
    assert lib.closed and r["source"].startswith("NVML")
    assert r["samples_in_window"] >= 5 and r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == ["sw_power_cap"] and r["power_w_max"] == 1380.0
    assert r["sm_mhz"] == 1700.0    # most samples sit at the last clock


def test_per_config_covers_every_specified_configuration():
    """C1, C2 (both masks), C3, C4 and C5 of the specification, each once."""
    shapes = {(w.B, w.H, w.Lq, w.Lk, w.D, w.causal)
              for w in (WORKLOADS[name] for _, name in bench.PER_CONFIG)}
    assert shapes == {(1, 2, 128, 128, 64, False), (4, 16, 1024, 1024, 64, False),
                      (4, 16, 1024, 1024, 64, True), (2, 32, 4096, 4096, 128, True),
                      (1, 16, 16384, 16384, 128, True), (8, 16, 500, 8191, 128, False)}
    assert len(bench.PER_CONFIG) == 6


def test_reference_arm_prints_the_contract_line():
    """The reference arm (the fp64 oracle on the host cores, a bounded row sample per step)
    prints one JSON line with the fields the benchmark contract asks of it; no GPU needed."""
    import os
    import subprocess
    import sys
    root = bench.ROOT
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--workload", "seq1k_d64_causal", "--steps", "1", "--warmup", "0",
                        "--ref-seconds-per-step", "0.5"],
                       capture_output=True, text=True, timeout=300, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "seq1k_d64_causal"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_under_two_ranks_prints_once():
    """Launched as two ranks (gloo on the CPU), only rank 0 times the oracle and prints; the
    other rank exits 0, and the oracle uses the host's cores despite the launcher's
    OMP_NUM_THREADS=1."""
    import os
    import subprocess
    import sys
    root = bench.ROOT
    env = dict(os.environ, BENCH_DIST_BACKEND="gloo")
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1", "--master-port", "29617",
                        os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--workload", "seq1k_d64_causal", "--steps", "1", "--warmup", "0",
                        "--ref-seconds-per-step", "0.5"],
                       capture_output=True, text=True, timeout=300, cwd=root, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    assert d["cpu_baseline"]["cores"] == cores
