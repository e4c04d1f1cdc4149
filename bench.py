"""Benchmark of the k-means assignment step on GB300 (one JSON line).

A step is one pass of the whole hot path over one batch of synthetic input:
centroid norms + assignment (one kmassign call with cnorm NULL, which forms
the norms inside; kmassign_norms ahead of the timing for the workload whose
norms are precomputed), inputs resident in HBM.  Default workload: N=262,144 points, D=256, K=16,384 centroids, X and C
iid N(0,1) in bf16 -- the shape the throughput target is stated on.

Metric: TFLOP/s counted as 2*N*K*D per step (the dense X.C^T the method
performs), whole job over all ranks.  Three seeded input sets rotate between
steps (410 MB in total, more than the 126 MB L2), as in the pages' method
(flashlib PR #22, "Benchmark methodology": three seeded sets rotated between
calls, warm-up calls, CUDA-event timing).  Workloads whose three sets fit in
twice the L2 get an L2 flush between timed steps instead (--l2).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload KEY]
  python bench.py --impl reference ...   # the fp64 CPU oracle, same metric

Multi-GPU (torchrun): every rank assigns its own batch of N points against
the full centroid set (points shard with no exchange), so scaling is weak;
the only collectives are the timing barrier and a max over ranks.
"""

from __future__ import annotations

import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "k-means assign TFLOP/s (2*N*K*D / t), 1 pass of norms + assignment"
UNIT = "TFLOP/s"
# The pages' own figure for this shape (B200, flashlib PR #22 "Benchmark
# results": N=262,144, D=256, K=16,384 in 1.8615 ms -> 1,181 TFLOP/s).
PAGES_B200_TFLOPS = {"iid_normal": 2 * 262144 * 16384 * 256 / 1.8615e-3 / 1e12}
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}
L2_BYTES_FALLBACK = 126 * 1024 * 1024    # GB300, when the device does not report it
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "assign_kernel_traffic.txt")


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, dist, device) -> float:
    """The largest of every rank's x (x itself without a process group)."""
    if dist is None or not dist.is_initialized():
        return float(x)
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_variants(rank: int, count: int = 3) -> list:
    """Seed variants of the rotating input sets of one rank (disjoint across ranks)."""
    return [count * int(rank) + v for v in range(count)]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def load_traffic(kernel_sha: str):
    """The ncu-measured DRAM bytes of one assign launch, if still current."""
    t = {}
    try:
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if line.startswith("#") or ":" not in line:
                    continue
                k, v = line.split(":", 1)
                v = v.strip()
                t[k.strip()] = int(v) if v.isdigit() else v
    except OSError:
        return None, None
    if not t:
        return None, None
    if t.get("source_sha") != kernel_sha:
        return None, t
    return t, t


# The sources assign_kernel is compiled from: a stored ncu traffic record is
# reported only while these are unchanged.
ASSIGN_KERNEL_SOURCES = [os.path.join("means_nearest_centroid_gb300", "csrc", f)
                         for f in ("assign.cu", "pipeline.cuh", "ptx.cuh", "internal.h")] + \
                        [os.path.join("include", "kmassign.h")]


def kernel_source_sha() -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in ASSIGN_KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(os.path.basename(rel).encode())
            h.update(f.read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        self.thread = None
        target = None
        try:
            props = torch.cuda.get_device_properties(device_index)
            uuid = getattr(props, "uuid", None)
            if uuid is not None:
                s = str(uuid)
                target = s if s.startswith("GPU-") else "GPU-" + s
        except Exception:
            target = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "20"]
        if target:
            cmd += ["-i", target]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                self.samples.append(dict(t=ts, sm=float(parts[1]), smax=float(parts[2]),
                                         power=float(parts[3]) if parts[3][0].isdigit() else None,
                                         hw=parts[4] == "Active", hwt=parts[5] == "Active",
                                         swt=parts[6] == "Active", pcap=parts[7] == "Active"))
            except (ValueError, IndexError):
                continue

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s["t"] <= t1]
        window = "timed"
        if not inside:
            inside = [s for s in self.samples if s["t"] <= t1 + 0.2]
            window = "warmup+timed"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window": "none"}
        reasons = set()
        for s in inside:
            if s["hw"]:
                reasons.add("hw_slowdown")
            if s["hwt"]:
                reasons.add("hw_thermal_slowdown")
            if s["swt"]:
                reasons.add("sw_thermal_slowdown")
            if s["pcap"]:
                reasons.add("sw_power_cap")
        return {"sm_mhz": statistics.median(s["sm"] for s in inside),
                "sm_max_mhz": max(s["smax"] for s in inside),
                "reasons": sorted(reasons), "samples": len(inside), "window": window}


class NvmlClockSampler:
    """The SM clock and the clock-event reasons read in-process through NVML
    (query calls only; nothing is set), every ~0.25 ms while running, so that
    even a timed region of a few tens of milliseconds gets many samples."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int):
        import ctypes
        self.samples = []
        self.ok = False
        self._stop = threading.Event()
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            handle = ctypes.c_void_p()
            uuid = str(getattr(torch.cuda.get_device_properties(device_index), "uuid", ""))
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(handle)) != 0:
                return
            self.lib, self.handle, self.ct = lib, handle, ctypes
            clk = ctypes.c_uint()
            if lib.nvmlDeviceGetClockInfo(handle, 1, ctypes.byref(clk)) != 0:   # 1: SM clock
                return
            mx = ctypes.c_uint()
            self.max_mhz = (float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(
                handle, 1, ctypes.byref(mx)) == 0 else None)
        except (OSError, AttributeError):
            return
        self.ok = True
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def _run(self):
        ct, lib, h = self.ct, self.lib, self.handle
        clk = ct.c_uint()
        rs = ct.c_ulonglong()
        while not self._stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ct.byref(clk)) == 0:
                r = (rs.value if lib.nvmlDeviceGetCurrentClocksEventReasons(h, ct.byref(rs)) == 0
                     else 0)
                self.samples.append((time.time(), float(clk.value), int(r)))
            time.sleep(0.00025)

    def stop(self):
        self._stop.set()
        if self.ok:
            self.thread.join(timeout=5)
            self.lib.nvmlShutdown()

    def by_clock(self, t0, intervals, flops, sms, bin_mhz=50.0):
        """Steps grouped by the SM clock seen while they ran: ``intervals``
        holds each step's (start, end) in seconds after the timed region began
        on the GPU (``t0`` in host time; the queue was empty then, so the GPU
        starts within microseconds).  Per bin of ``bin_mhz``: the steps, their
        mean kernel time and the rate per SM clock, so that a clock-bound and
        a clock-independent limit can be told apart within one run."""
        if not self.samples:
            return None
        import bisect
        ts = [s[0] for s in self.samples]
        bins = {}
        for a, b in intervals:
            i, j = bisect.bisect_left(ts, t0 + a), bisect.bisect_right(ts, t0 + b)
            mhz = [self.samples[k][1] for k in range(i, j)]
            if not mhz:   # no sample inside this step: the nearest one
                k = min(max(i, 0), len(ts) - 1)
                mhz = [self.samples[k][1]]
            m = statistics.mean(mhz)
            bins.setdefault(round(m / bin_mhz) * bin_mhz, []).append((b - a, m))
        out = []
        for c in sorted(bins):
            v = bins[c]
            ms = statistics.mean(d for d, _ in v) * 1e3
            mhz = statistics.mean(m for _, m in v)
            out.append({"sm_mhz": round(mhz), "steps": len(v), "kernel_ms": round(ms, 4),
                        "tflops": round(flops / (ms * 1e-3) / 1e12, 1),
                        "flop_per_clk_per_sm": round(flops / (ms * 1e-3) / (sms * mhz * 1e6))})
        return out

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        if not inside:
            return None
        reasons = sorted({name for _, _, r in inside for bit, name in self.REASONS.items()
                          if r & bit})
        mhz = [m for _, m, _ in inside]
        return {"sm_mhz": statistics.median(mhz), "sm_mhz_min": min(mhz), "sm_mhz_max": max(mhz),
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(inside),
                "source": "NVML in-process, every ~0.25 ms over the timed steps"}


def make_inputs(key, variants, device, N=None, K=None, D=None):
    sets = []
    for v in variants:
        X, C = workloads.make(key, N=N, K=K, D=D, variant=v)
        sets.append((X, C))
    dev_sets = [(X.to(device), C.to(device)) for X, C in sets]
    return sets, dev_sets


def cpu_oracle_rate(X, C, budget_s: float, max_rows: int | None = None):
    """Time the fp64 oracle on the first R rows of X against all of C.

    R is picked from a short calibration so the measured run takes about
    budget_s seconds.  Returns (tflops, rows, seconds, threads).
    """
    import oracle
    orc = oracle.Oracle()
    threads = orc.max_threads()
    K, D = C.shape
    cn = orc.norms(C)
    probe = max(threads, 8)
    t0 = time.perf_counter()
    orc.assign(X[:probe], C, cnorm=cn)
    dt = time.perf_counter() - t0
    per_row = dt / probe
    rows = int(max(threads, min(X.shape[0], budget_s / max(per_row, 1e-9))))
    if max_rows:
        rows = min(rows, max_rows)
    t0 = time.perf_counter()
    orc.assign(X[:rows], C, cnorm=cn)
    dt = time.perf_counter() - t0
    return 2.0 * rows * K * D / dt / 1e12, rows, dt, threads


def run_reference(args, key):
    """The fp64 CPU oracle as the reference arm, same metric and config."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = workloads.WORKLOADS[key]
    X, C = workloads.make(key)
    import oracle
    orc = oracle.Oracle()
    threads = orc.max_threads()
    cn = orc.norms(C)
    probe = max(threads, 8)
    t0 = time.perf_counter()
    orc.assign(X[:probe], C, cnorm=cn)
    per_row = (time.perf_counter() - t0) / probe
    total_budget = args.ref_budget_s
    per_step = total_budget / max(1, args.steps + args.warmup)
    rows = int(max(threads, min(w.N, per_step / max(per_row, 1e-9))))
    for _ in range(args.warmup):
        orc.assign(X[:rows], C, cnorm=cn)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        orc.assign(X[:rows], C, cnorm=cn)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = 2.0 * rows * w.K * w.D * args.steps / total / 1e12
    sample = (f"first {rows} of {w.N} points against all {w.K} centroids per step "
              f"(fp64 oracle, OpenMP over points)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.text, "key": key, "N": w.N, "D": w.D, "K": w.K,
                   "sample_rows": rows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# The 13 shapes of the pages' benchmark (flashlib PR #22, Performance and
# "Benchmark results" tables) with their B200 latencies, context only.
PAGES_SHAPES = [  # N, D, K, nightly ms, PR ms (B200)
    (65536, 64, 512, 0.0727, 0.0441), (65536, 64, 4096, 0.1332, 0.1022),
    (65536, 64, 16384, 0.3462, 0.2963), (65536, 128, 512, 0.0722, 0.0453),
    (65536, 128, 4096, 0.1399, 0.1059), (262144, 128, 4096, 0.3444, 0.2844),
    (262144, 128, 16384, 1.1653, 1.0047), (1048576, 128, 4096, 1.1978, 1.0148),
    (65536, 256, 512, 0.0871, 0.0587), (65536, 256, 4096, 0.2111, 0.1661),
    (262144, 256, 4096, 0.5640, 0.4631), (262144, 256, 16384, 2.0881, 1.8615),
    (1048576, 256, 4096, 2.1431, 1.9458),
]


def run_pages_shapes(device):
    """The pages' 13 shapes on this GPU, their method: three seeded bf16 sets
    (17, 29, 43) rotated between calls, 10 warm-up and 30 timed calls, CUDA
    events, median.  iid N(0,1) inputs (the pages give no distribution); norms
    precomputed, so the time is the assignment call.  One JSON line each."""
    import means_nearest_centroid_gb300 as km
    stream = torch.cuda.current_stream(device)
    rows = []
    for N, D, K, nightly, pr in PAGES_SHAPES:
        sets = []
        for seed in (17, 29, 43):
            X, C = workloads.iid(N, K, D, seed)
            Xd, Cd = X.to(device), C.to(device)
            sets.append((Xd, Cd, km.kmassign_norms(Cd, stream=stream),
                         torch.empty(N, dtype=torch.int32, device=device)))
        for i in range(10):
            Xd, Cd, cn, idx = sets[i % 3]
            km.kmassign(Xd, Cd, cnorm=cn, idx=idx, stream=stream)
        times = []
        for i in range(30):
            Xd, Cd, cn, idx = sets[i % 3]
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            km.kmassign(Xd, Cd, cnorm=cn, idx=idx, stream=stream)
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
        rc = km.kmassign_check(stream)
        ms = statistics.median(times)
        line = {"N": N, "D": D, "K": K, "ms": ms, "tflops": 2.0 * N * K * D / ms / 1e9,
                "b200_pr_ms": pr, "b200_nightly_ms": nightly, "status": rc,
                "plan": km.kmassign_plan(N, K, D)}
        rows.append(line)
        print(json.dumps(line), flush=True)
        del sets
    geo = statistics.geometric_mean([r["ms"] for r in rows])
    print(json.dumps({"geomean_ms": geo,
                      "b200_pr_geomean_ms": statistics.geometric_mean([r[4] for r in PAGES_SHAPES]),
                      "b200_nightly_geomean_ms": statistics.geometric_mean([r[3] for r in PAGES_SHAPES])}),
          flush=True)
    return 0


def run_update_bench(device, key, steps, warmup):
    """The update step (kmassign_update) on a workload, against the HBM roofline,
    and one whole Lloyd iteration (norms + assignment + update + centroids).
    Three rotating input sets, as in the main benchmark.  One JSON line."""
    import means_nearest_centroid_gb300 as km
    w = workloads.WORKLOADS[key]
    N, D, K = w.N, w.D, w.K
    stream = torch.cuda.current_stream(device)
    sets = []
    for v in range(3):
        X, C = workloads.make(key, variant=v)
        Xd, Cd = X.to(device), C.to(device)
        sets.append((Xd, Cd, km.kmassign(Xd, Cd, stream=stream)))
    sums = torch.zeros((K, D), dtype=torch.float32, device=device)
    counts = torch.zeros(K, dtype=torch.int32, device=device)
    def time_update(method):
        for i in range(warmup):
            Xd, Cd, idx = sets[i % 3]
            km.kmassign_update(Xd, idx, K, sums=sums, counts=counts, method=method, stream=stream)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for i in range(steps):
            Xd, Cd, idx = sets[i % 3]
            sums.zero_()
            counts.zero_()
            evs[i][0].record(stream)
            km.kmassign_update(Xd, idx, K, sums=sums, counts=counts, method=method, stream=stream)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in evs)

    method_ms = {"atomic": time_update(1), "sorted": time_update(2)}
    upd_ms = time_update(0)
    peaks, src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    alg_bytes = 2 * N * D + 4 * N + 8 * K * D + 4 * K
    # a whole iteration on the device
    Cw = sets[0][1].clone()
    km.kmassign_lloyd(sets[0][0], Cw, iters=2, stream=stream)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    km.kmassign_lloyd(sets[0][0], Cw, iters=steps, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    it_ms = e0.elapsed_time(e1) / steps
    rc = km.kmassign_check(stream)
    line = {"metric": "k-means update step GB/s (algorithmic bytes / t) and Lloyd iteration ms",
            "value": alg_bytes / (upd_ms * 1e-3) / 1e9, "unit": "GB/s", "steps": steps,
            "warmup": warmup, "higher_is_better": True, "dtype": "bf16 in, fp32 sums",
            "data": "synthetic", "status": rc,
            "config": {"workload": w.text, "key": key, "N": N, "D": D, "K": K},
            "update_ms": upd_ms, "update_ms_by_method": method_ms,
            "roofline": {"bound": "hbm", "achieved": alg_bytes / (upd_ms * 1e-3) / 1e9,
                         "peak": hbm, "unit": "GB/s",
                         "frac": alg_bytes / (upd_ms * 1e-3) / 1e9 / hbm,
                         "peak_source": f"{src} copy bandwidth", "traffic": None,
                         "algorithmic_bytes": alg_bytes},
            "lloyd_iteration_ms": it_ms,
            "lloyd_iteration_tflops": 2.0 * N * K * D / (it_ms * 1e-3) / 1e12}
    print(json.dumps(line), flush=True)
    return 0


def run_topk_bench(device, key, ks, steps, warmup, distances=False, sizes=(None, None, None)):
    """The k-nearest call (kmassign_topk) for each k in ``ks`` on a workload,
    beside the assignment (kmassign) on the same three rotating input sets,
    norms precomputed so both times are the kernel calls.  One JSON line per k;
    the roofline is the tensor-pipe bound of the same 2*N*K*D contraction."""
    import means_nearest_centroid_gb300 as km
    w = workloads.WORKLOADS[key]
    N = sizes[0] or w.N
    K = sizes[1] or w.K
    D = sizes[2] or w.D
    stream = torch.cuda.current_stream(device)
    sets = []
    for v in range(3):
        X, C = workloads.make(key, N=N, K=K, D=D, variant=v)
        Xd, Cd = X.to(device), C.to(device)
        sets.append((Xd, Cd, km.kmassign_norms(Cd, stream=stream)))
    peaks, src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))

    def timed(call):
        for i in range(warmup):
            call(*sets[i % 3])
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for i in range(steps):
            evs[i][0].record(stream)
            call(*sets[i % 3])
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in evs)

    idx1 = torch.empty(N, dtype=torch.int32, device=device)
    base_ms = timed(lambda Xd, Cd, cn: km.kmassign(Xd, Cd, cnorm=cn, idx=idx1, stream=stream))
    flops = 2.0 * N * K * D
    for k in ks:
        idx = torch.empty((N, k), dtype=torch.int32, device=device)
        sc = torch.empty((N, k), dtype=torch.float32, device=device)
        ms = timed(lambda Xd, Cd, cn: km.kmassign_topk(Xd, Cd, k, cnorm=cn, idx=idx, score=sc,
                                                       distances=distances, stream=stream))
        rc = km.kmassign_check(stream)
        tf = flops / (ms * 1e-3) / 1e12
        line = {"metric": "k nearest centroids, TFLOP/s of the score contraction",
                "value": tf, "unit": "TFLOP/s", "k": k, "distances": distances,
                "ms": ms, "assign_ms": base_ms, "vs_assign": base_ms / ms,
                "steps": steps, "warmup": warmup, "higher_is_better": True,
                "dtype": "bf16 in, fp32 scores", "data": "synthetic", "status": rc,
                "config": {"workload": w.text if (N, K, D) == (w.N, w.K, w.D) else
                           f"{key} recipe at N={N}, K={K}, D={D}", "key": key, "N": N, "D": D,
                           "K": K, "l2": "3 rotating input sets"},
                "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                             "frac": tf / peak, "peak_source": f"{src} bf16 burst"}}
        print(json.dumps(line), flush=True)
        del idx, sc
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="iid_normal", choices=list(workloads.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--ref-budget-s", type=float, default=150.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pages-shapes", action="store_true",
                    help="time the pages' 13 benchmark shapes instead (context table)")
    ap.add_argument("--update", action="store_true",
                    help="time the update step and a Lloyd iteration instead")
    ap.add_argument("--topk", default=None,
                    help="comma-separated k values: time the k-nearest call instead")
    ap.add_argument("--distances", action="store_true",
                    help="with --topk: write squared distances instead of scores")
    ap.add_argument("--l2", default="auto", choices=["auto", "flush", "none"],
                    help="flush L2 between timed steps: auto = when the rotating inputs do not "
                         "exceed twice the L2")
    ap.add_argument("--parity-rows", type=int, default=256)
    ap.add_argument("--N", type=int, default=None, help="override the workload's N")
    ap.add_argument("--K", type=int, default=None, help="override the workload's K")
    ap.add_argument("--D", type=int, default=None, help="override the workload's D")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    key = args.workload
    if args.impl == "reference":
        return run_reference(args, key)

    ws, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (there is no CPU path)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if args.pages_shapes or args.update or args.topk:
        from means_nearest_centroid_gb300 import _build
        _build.build()
        if args.pages_shapes:
            return run_pages_shapes(device)
        if args.topk:
            ks = [int(v) for v in args.topk.split(",")]
            return run_topk_bench(device, key, ks, args.steps, args.warmup, args.distances,
                                  (args.N, args.K, args.D))
        return run_update_bench(device, key, args.steps, args.warmup)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    else:
        dist = None

    from means_nearest_centroid_gb300 import _build
    if rank == 0:
        _build.build()
    if dist is not None:
        dist.barrier()
    import means_nearest_centroid_gb300 as km
    km.library()

    w = workloads.WORKLOADS[key]
    N = w.N if args.N is None else args.N
    D = w.D if args.D is None else args.D
    K = w.K if args.K is None else args.K
    resized = (N, D, K) != (w.N, w.D, w.K)
    flops = 2.0 * N * K * D
    sets, dsets = make_inputs(key, rank_variants(rank), device, N, K, D)
    cns = [torch.empty(K, dtype=torch.float32, device=device) for _ in dsets]
    idxs = [torch.empty(N, dtype=torch.int32, device=device) for _ in dsets]
    stream = torch.cuda.current_stream(device)
    plan = km.kmassign_plan(N, K, D)
    norms_in_step = not w.precomputed_norms
    if not norms_in_step:
        for (X, C), cn in zip(dsets, cns):
            km.kmassign_norms(C, out=cn, stream=stream)

    # L2: the three rotating sets together must exceed L2 between timed steps;
    # when they do not (the small workloads), a buffer larger than L2 is
    # written between steps, outside the steps' own events.
    l2_bytes = int(getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 0)) or \
        L2_BYTES_FALLBACK
    set_bytes = sum(X.numel() * 2 + C.numel() * 2 + N * 4 + K * 4 for X, C in dsets)
    flush = args.l2 == "flush" or (args.l2 == "auto" and set_bytes < 2 * l2_bytes)
    flush_buf = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=device) if flush else None

    def step(i, ev_mid=None, ev_end=None, ev_begin=None):
        # norms in the step: one call with cnorm NULL, which computes them
        # inside (in the same launch that prepares the call's other inputs)
        X, C = dsets[i % 3]
        if flush_buf is not None:
            flush_buf.fill_(i & 0xff)
        if ev_begin is not None:
            ev_begin.record(stream)
        if ev_mid is not None:
            ev_mid.record(stream)
        km.kmassign(X, C, cnorm=None if norms_in_step else cns[i % 3], idx=idxs[i % 3],
                    stream=stream)
        if ev_end is not None:
            ev_end.record(stream)

    sampler = ClockSampler(local)
    nvml = NvmlClockSampler(local)
    time.sleep(0.3)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    rc = km.kmassign_check(stream)
    if rc != 0:
        raise SystemExit(f"warm-up failed: {km.kmassign_strerror(rc)}")

    begins = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_stop = torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    t_start.record(stream)
    for i in range(args.steps):
        step(i, mids[i], ends[i], begins[i])
    t_stop.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    if dist is not None:
        dist.barrier()
    rc = km.kmassign_check(stream)
    if rc != 0:
        raise SystemExit(f"timed run failed: {km.kmassign_strerror(rc)}")
    sampler.stop()
    nvml.stop()
    total_ms = t_start.elapsed_time(t_stop)
    kern_ms = [m.elapsed_time(e) for m, e in zip(mids, ends)]
    if flush_buf is not None:
        # the flushes sit between the steps: count the steps' own time only
        total_ms = sum(b.elapsed_time(e) for b, e in zip(begins, ends))
    total_ms = max_over_ranks(total_ms, dist, device)
    ms_per_step = total_ms / args.steps
    value = flops * ws * args.steps / (total_ms * 1e-3) / 1e12

    # ---- roofline of the dominant kernel (the assignment kernel)
    peaks, peak_src = load_peaks()
    kernel_avg_ms = statistics.mean(kern_ms)
    kernel_med_ms = statistics.median(kern_ms)
    achieved = flops / (kernel_avg_ms * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sha = kernel_source_sha()
    traffic, traffic_rec = load_traffic(sha)
    pair = plan["rows_per_cta"] == 256 and plan["centroids_per_tile"] == 256
    tile = f'{plan["rows_per_cta"]}x{plan["centroids_per_tile"]}{" pair" if pair else ""}'
    traffic_bytes = None
    if (traffic is not None and not resized and traffic.get("workload") == key
            and traffic.get("tile") == tile):
        traffic_bytes = traffic.get("bytes_per_launch")
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic_bytes,
                "peak_source": f"{peak_src} bf16 dense (burst)",
                "kernel": ("assign_pair_kernel (tcgen05.cta_group::2, " if pair
                           else "assign_kernel (tcgen05, ") + tile + " tiles)",
                "timed": "the kmassign call around the kernel (its preparation launch, when "
                         "one runs, included), CUDA events on the launching stream",
                "kernel_ms_avg": kernel_avg_ms,
                "kernel_ms_median": kernel_med_ms,
                "algorithmic_bytes": N * D * 2 + K * D * 2 + N * 4 + K * 4}

    # ---- parity sample against the oracle (rows computed one by one)
    parity_info = None
    if rank == 0 and args.parity_rows > 0:
        import oracle
        orc = oracle.Oracle()
        X0, C0 = sets[0]
        g = np.random.default_rng(w.seed)
        rows = np.sort(g.choice(N, min(N, args.parity_rows), replace=False))
        idx0 = idxs[0].cpu().numpy().astype(np.int64)
        o_idx, o_min = orc.assign(X0, C0, rows=rows)
        diff = np.nonzero(idx0[rows] != o_idx)[0]
        bad = 0
        if diff.size:
            s = orc.scores(X0, C0, rows[diff], idx0[rows][diff])
            xs = X0[rows[diff]].double().numpy()
            scale = (xs * xs).sum(1) + orc.norms(C0)[idx0[rows][diff]]
            bad = int(np.sum(~(s - o_min[diff] <= 2e-5 * scale)))
        parity_info = {"rows": int(rows.size), "idx_differs": int(diff.size),
                       "outside_tolerance": bad}

    # ---- end to end through the C ABI with host buffers (kmassign_host)
    e2e = None
    if args.e2e_steps > 0:
        X0, C0 = sets[0]
        Xh = X0.pin_memory()
        Ch = C0.pin_memory()
        cnh = None if norms_in_step else cns[0].cpu().pin_memory()
        idx_h = torch.empty(N, dtype=torch.int32).pin_memory()
        km.assign_host(Xh, Ch, idx_h, cnorm_host=cnh, device=device)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            km.assign_host(Xh, Ch, idx_h, cnorm_host=cnh, device=device)
        e2e_s = max_over_ranks(time.perf_counter() - t0, dist, device)
        h2d = Xh.numel() * 2 + Ch.numel() * 2 + (0 if cnh is None else cnh.numel() * 4)
        e2e = {"value": flops * ws * args.e2e_steps / e2e_s / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": idx_h.numel() * 4, "steps": args.e2e_steps,
               "ms_per_step": 1e3 * e2e_s / args.e2e_steps,
               "note": "every step one kmassign_host call (C ABI, pinned host buffers): C"
                       + ("" if cnh is None else " and its norms") + " copied in, X in row "
                       "slices of whole waves overlapped with the assignment of the previous "
                       "slice, " + ("norms + " if cnh is None else "") + "assignment, idx "
                       "copied out per slice; the call returns when idx is in host memory"}

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N=1 only)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        X0, C0 = sets[0]
        rate, rows, secs, threads = cpu_oracle_rate(X0, C0, args.cpu_budget_s)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"first {rows} of {N} points against all {K} centroids, "
                         f"{secs:.1f} s, fp64 oracle (OpenMP over points)"}

    clocks = sampler.summary(wall0, wall1)
    nv = nvml.summary(wall0, wall1)
    if nv is not None and nv["samples"] >= 5:
        smi = clocks
        clocks = dict(nv)
        clocks["reasons"] = sorted(set(nv["reasons"]) | set(smi.get("reasons", [])))
        clocks["nvidia_smi"] = smi
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    if clocks.get("sm_mhz"):
        # clock-normalised rate of the dominant kernel: flop per SM clock
        roofline["flop_per_clk_per_sm"] = achieved * 1e12 / (sms * clocks["sm_mhz"] * 1e6)
        roofline["sms"] = sms
    if nvml.ok:
        # each step's kernel interval on the GPU, paired with the clock then
        spans = [(t_start.elapsed_time(m) * 1e-3, t_start.elapsed_time(e) * 1e-3)
                 for m, e in zip(mids, ends)]
        binned = nvml.by_clock(wall0, spans, flops, sms)
        if binned:
            clocks["by_clock"] = binned
    # the preparation launch (norms when computed in the step, the fold
    # operand of a CTA pair folding the norms at D <= 128, the split rows'
    # keys) and the assignment kernel, which also finalizes split rows
    folding_pair = pair and D <= 128
    prep = norms_in_step or folding_pair or plan["ksplit"] > 1
    launches_per_step = (1 if prep else 0) + 1
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": (value / PAGES_B200_TFLOPS[key])
        if (key in PAGES_B200_TFLOPS and not resized) else None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": (f"{key} distribution resized to N={N}, D={D}, K={K}"
                                if resized else w.text), "key": key, "N": N, "D": D, "K": K,
                   "norms_in_step": norms_in_step,
                   "l2": (f"L2 ({l2_bytes / 2**20:.0f} MiB) flushed between timed steps by "
                          f"writing {2 * l2_bytes / 2**20:.0f} MiB outside the steps' events; "
                          f"3 rotating sets of {set_bytes / 2**20:.0f} MiB in total"
                          if flush_buf is not None else
                          f"3 rotating seeded input sets per GPU, {set_bytes / 2**20:.0f} MiB "
                          f"together, larger than twice the {l2_bytes / 2**20:.0f} MiB L2"
                          if set_bytes >= 2 * l2_bytes else
                          f"not flushed (--l2 none): 3 rotating sets of {set_bytes / 2**20:.0f} "
                          f"MiB may stay in the {l2_bytes / 2**20:.0f} MiB L2"),
                   "plan": plan, "parallelism": f"points sharded, {ws} independent batches"},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "parity_sample": parity_info,
    }
    if traffic_rec is not None and traffic_bytes is None:
        line["roofline"]["traffic_note"] = "stored ncu traffic is for another kernel revision or workload"
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
