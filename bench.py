"""Benchmark of the fine-grained FP8 path on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--rows all|none]
    python bench.py --case NAME [--reps R]     (one kernel on a bounded case, for ncu captures)

One step = one pass of the dense-linear workload through the whole path:
1x128 quantisation of X [4096, 7168] and 128x128 quantisation of W [7168,
7168] (one launch), then the block-scaled FP8 GEMM -> bf16 Y [4096, 7168]
(a programmatic dependent launch), inputs resident in HBM.  The headline
value is the step's GEMM FLOPs / step time (TFLOP/s).
Between timed steps L2 is flushed (outside each step's events): a 256 MiB
buffer is written and then read back, so that L2 holds only clean lines of
it and the next kernel starts cold without paying for dirty write-backs.  Rank 0 prints one JSON line.

Besides the headline, ``rows`` times every step of the path on its own
workload (the 128x1 quantiser and Wgrad GEMM, the grouped MoE GEMMs, routing,
dispatch and combine) against its roofline.

With N > 1 (torchrun) every rank runs the same workload independently: the
path has no exchange step on one GPU, so this is N replicas (weak scaling);
the step time is the max over ranks.

``--impl reference`` times the CPU oracle (the plain definition of what the
path computes) on a bounded sample of the same workload, on rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

M, N, K = 4096, 7168, 7168
GEMM_FLOP = 2.0 * M * N * K
FP8_NOMINAL_TFLOPS = 4500.0           # dense E4M3, nominal
HBM_NOMINAL_GBS = 8000.0
METRIC = "FP8 block-scaled GEMM TFLOP/s (% FP8 peak); quantize GB/s (% HBM peak)"
WORKLOAD = ("dense linear: X bf16 [4096,7168] ~0.5*t(3), W bf16 [7168,7168] ~N(0,0.02^2); "
            "quantise X 1x128 + quantise W 128x128 + block-scaled FP8 GEMM -> bf16 [4096,7168]")


# ---------------------------------------------------------------- helpers
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), src="measured")
    return dict(hbm=6400.0, bf16=1800.0, bf16_sustained=1400.0, src="fallback")


def max_over_ranks(x: float, ws: int, device=None) -> float:
    """The largest per-rank value (time per step): the job is as slow as its
    slowest rank."""
    if ws <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, ws: int, ms: float) -> float:
    """Whole-job rate: the units every rank processed per second of the
    slowest rank's step time."""
    return units_per_rank * ws / (ms * 1e-3)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Clocks:
    """nvidia-smi sampled every 100 ms while the timed region runs."""

    def __init__(self, index: int):
        self.index = index
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        self.proc = None

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        # nvidia-smi needs a moment to start: wait for its first sample so the
        # timed region is covered from its start; samples taken before
        # t_start are dropped in summary().
        t0 = time.time()
        while self.proc and time.time() - t0 < 10.0 and self.proc.poll() is None:
            self.f.flush()
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)
        self.skip = self._lines()
        self.t_start = time.time()
        return self

    def _lines(self):
        try:
            return sum(1 for _ in open(self.path))
        except OSError:
            return 0

    def __exit__(self, *a):
        if self.proc:
            # let at least one sample land inside a short timed region
            time.sleep(max(0.0, 0.25 - (time.time() - self.t_start)))
            self.proc.terminate()
            self.proc.wait()
            self.f.close()

    def summary(self):
        if not self.proc:
            return None
        rows = []
        for i, line in enumerate(open(self.path)):
            if i < self.skip:
                continue
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smax=float(f[2]), power=float(f[3]),
                                 hw=f[5] == "Active", hwt=f[6] == "Active", swt=f[7] == "Active",
                                 cap=f[8] == "Active"))
            except ValueError:
                pass
        os.unlink(self.path)
        if not rows:
            return None
        reasons = []
        for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                          ("swt", "sw_thermal_slowdown"), ("cap", "sw_power_cap")):
            if any(r[key] for r in rows):
                reasons.append(name)
        return dict(sm_mhz=statistics.median(r["sm"] for r in rows), sm_mhz_min=min(r["sm"] for r in rows),
                    sm_max_mhz=max(r["smax"] for r in rows), reasons=reasons, samples=len(rows),
                    power_w_max=max(r["power"] for r in rows))


class L2Flush:
    """Evict L2 between timed steps: write a buffer twice the size of L2, then
    read it back (a sum), which writes the dirty lines back to HBM and leaves
    L2 full of clean lines that the next kernel can drop for free."""

    def __init__(self, dev, nbytes=256 << 20):
        self.buf = torch.empty(nbytes // 8, dtype=torch.int64, device=dev)
        self.sink = torch.empty((), dtype=torch.int64, device=dev)

    def __call__(self):
        self.buf.zero_()
        torch.sum(self.buf, dim=0, out=self.sink)


def kernel_source_sha():
    """Hash of the GEMM's code (its .cu and the headers it includes), with
    `//` comments and blank lines left out, so that a comment edit keeps a
    traffic record taken on the same code."""
    h = hashlib.sha256()
    for f in ("gemm.cu", "common.cuh", "tail_split.cuh", "expert_sched.cuh", "tensor_map.cuh"):
        for line in open(os.path.join(ROOT, "fp8_fine_grained_16_b300", "csrc", f)):
            code = line.split("//", 1)[0].rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def ncu_traffic():
    """DRAM bytes per launch of the dense-linear GEMM from the committed ncu
    summary, if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "gemm_dense_linear_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("kernel_src_sha") != kernel_source_sha():
        return None
    return d.get("dram_bytes_per_launch")


def link_time(x_h, w_h, y_h, x, w, y, stream, reps=5):
    """The host link's own time for one step's bytes: X and W host->device
    beside Y device->host, on two streams, nothing else (best of `reps`).
    This bounds the end-to-end step: the copies in the two directions share
    the link, so they take longer together than the one-way copy in."""
    a, b = torch.cuda.Stream(stream.device), torch.cuda.Stream(stream.device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = float("inf")
    for _ in range(reps):
        torch.cuda.synchronize()
        e0.record(stream)
        a.wait_stream(stream)
        b.wait_stream(stream)
        with torch.cuda.stream(a):
            x.copy_(x_h, non_blocking=True)
            w.copy_(w_h, non_blocking=True)
        with torch.cuda.stream(b):
            y_h.copy_(y, non_blocking=True)
        stream.wait_stream(a)
        stream.wait_stream(b)
        e1.record(stream)
        e1.synchronize()
        best = min(best, e0.elapsed_time(e1))
    return best


# ---------------------------------------------------------------- our arm
def run_ours(args, ws, rank, local):
    from fp8_fine_grained_16_b300 import build
    build.build()
    from fp8_fine_grained_16_b300 import fp8bs as F
    from fp8_fine_grained_16_b300 import synthetic as S

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    pk = peaks()

    d = S.dense_linear()
    x_h, w_h = d["x"].pin_memory(), d["w"].pin_memory()
    x, w = x_h.to(dev), w_h.to(dev)
    qx = torch.empty((M, K), dtype=torch.uint8, device=dev)
    sx = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
    qw = torch.empty((N, K), dtype=torch.uint8, device=dev)
    sw = torch.empty((N // 128, K // 128), dtype=torch.float32, device=dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    flush = L2Flush(dev)

    # The two quantisers are independent HBM-bound passes: one launch runs both
    # (X's 1x128 rows and W's 128x128 blocks side by side), and the GEMM after
    # it is a programmatic dependent launch that sets up while they drain.
    def step(evs=None):
        if evs:
            evs[0].record(stream)
        F.fp8_quant_act_weight(x, w, qx, sx, qw, sw)
        if evs and len(evs) == 3:
            evs[1].record(stream)           # breaks the programmatic overlap: only in the GEMM's own pass
        F.fp8_gemm_blockscaled(qx, sx, qw, sw, 0, torch.bfloat16, d=y)
        if evs:
            evs[-1].record(stream)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    if F.fp8_get_status() != 0:
        raise RuntimeError("device status set during warm-up")

    def timed_steps(n, marks):
        """n steps back to back on the GPU (flush, step, flush, step, ...; no
        host synchronisation inside), each bracketed by `marks` events."""
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(marks)] for _ in range(n)]
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        # a device-side sleep first, so the host enqueues ahead of the GPU and
        # no step's events include host launch time
        torch.cuda._sleep(50_000_000)
        for i in range(n):
            flush()
            step(evs[i])
        torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        return evs

    # Timed region: the steps as they run, events only at their ends.
    with Clocks(local) as clk:
        evs = timed_steps(args.steps, 2)
    t_step = [e[0].elapsed_time(e[1]) for e in evs]
    if F.fp8_get_status() != 0:
        raise RuntimeError("device status set during the timed steps")
    ms = max_over_ranks(sum(t_step) / len(t_step), ws, dev)
    clocks = clk.summary()
    # The GEMM's own duration (the roofline's denominator): the same steps
    # again with an event between the quantisers and the GEMM, which makes the
    # GEMM wait for them and so times its whole launch, set-up included.
    n_split = min(args.steps, 200)
    evs3 = timed_steps(n_split, 3)
    t_q = [e[0].elapsed_time(e[1]) for e in evs3]
    t_gemm = [e[1].elapsed_time(e[2]) for e in evs3]
    if F.fp8_get_status() != 0:
        raise RuntimeError("device status set during the timed steps")
    gemm_ms = sum(t_gemm) / len(t_gemm)
    q_ms = sum(t_q) / len(t_q)
    fp8_peak = pk["bf16"] * 2.0             # E4M3 dense = 2x bf16 dense (nominal 4.5 / 2.25 PFLOP/s)
    achieved = GEMM_FLOP / (gemm_ms * 1e-3) / 1e12

    # ---- end to end through the C-ABI call that takes HOST buffers: X and W
    # from pinned host memory, Y back to pinned host memory, every copy inside
    # the events (fp8_linear_host overlaps them with the GPU work by chunks)
    y_h = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ms = []
    e2e_steps = min(args.steps, 30)
    for i in range(args.warmup + e2e_steps):
        flush()
        torch.cuda.synchronize()
        e_start.record(stream)
        F.fp8_linear_host(x_h, w_h, y_h)
        e_end.record(stream)
        e_end.synchronize()
        if i >= args.warmup:
            e2e_ms.append(e_start.elapsed_time(e_end))
    e2e = sum(e2e_ms) / len(e2e_ms)
    if F.fp8_get_status() != 0:
        raise RuntimeError("device status set during the end-to-end steps")
    link = link_time(x_h, w_h, y_h, x, w, y, stream)

    rows = rows_clocks = None
    if args.rows != "none":
        sections = None if args.rows == "all" else tuple(x for x in args.rows.split(",") if x)
        # clocks sampled over the whole row measurement, so that a row run at a
        # lower SM clock shows (the step's own clocks are in "clocks")
        with Clocks(local) as clk_rows:
            rows = measure_rows(F, S, dev, flush, pk) if sections is None else \
                measure_rows(F, S, dev, flush, pk, sections)
        rows_clocks = clk_rows.summary()

    out = {
        "metric": METRIC,
        "value": round(job_throughput(GEMM_FLOP, ws, ms) / 1e12, 2),
        "unit": "TFLOP/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 (fp32 accumulate, bf16 out)",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "l2": "flushed between steps (256 MiB write + read-back)",
                   "parallelism": "replicas" if ws > 1 else "single GPU"},
        "roofline": {"bound": "tensor",
                     "kernel": "gemm_pair_kernel + splitk_fixup_kernel (dense linear 4096x7168x7168)",
                     "achieved": round(achieved, 1), "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                     "frac": round(achieved / fp8_peak, 4),
                     "peak_source": "%s bf16 burst x 2 (E4M3/bf16 nominal ratio)" % pk["src"],
                     "frac_of_nominal_4500": round(achieved / FP8_NOMINAL_TFLOPS, 4),
                     "traffic": ncu_traffic()},
        "step_breakdown_ms": {"quant_act_and_weight_one_launch": round(q_ms, 5),
                              "gemm": round(gemm_ms, 5),
                              "timed_apart_steps": n_split,
                              "how": "a second pass of the same steps with an event between the two launches; "
                                     "the timed steps themselves have none, so the GEMM's set-up overlaps "
                                     "the quantisers there"},
        "e2e": {"value": round(GEMM_FLOP * ws / (e2e * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "ms_per_step": round(e2e, 4), "steps": e2e_steps,
                "api": "fp8_linear_host: pinned host X, W -> pinned host Y, copies chunked and overlapped",
                "link_ms": round(link, 4), "frac_of_link": round(link / e2e, 4),
                "h2d_bytes_per_step": x.numel() * 2 + w.numel() * 2, "d2h_bytes_per_step": y.numel() * 2},
        # quant_act_weight (X and W), the GEMM and (when it splits its last wave) its fix-up
        "gpu_launches": (1 + gemm_launches(F, M, N, K, dev)) * args.steps,
        "clocks": clocks,
    }
    if rows is not None:
        out["rows"] = rows
        out["rows_clocks"] = rows_clocks
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(S, d=d, dev=dev)
    return out


def gemm_launches(F, m, n, k, dev) -> int:
    """Kernels one fp8_gemm_blockscaled call (with its workspace) launches: the
    GEMM, plus the fix-up kernel when the library's plan splits the last wave
    along K (256-row tiles on one SM pair each)."""
    pairs = torch.cuda.get_device_properties(dev).multi_processor_count // 2
    split, _, _ = F.fp8_gemm_split_plan(m, n, k, pairs, F.lib.fp8_gemm_blockscaled_workspace_bytes(m, n, k))
    return 2 if split > 0 else 1


class _SmClock:
    """The SM clock read through NVML right after each timed repetition, so
    that every row carries the clock it ran at (a row measured at a lower
    clock -- the power cap acting after the heavy rows -- shows as such).
    NVML comes from pynvml if installed, else from the driver's
    libnvidia-ml.so.1 through ctypes; without either, one nvidia-smi query
    per row stands in."""

    def __init__(self):
        self.h = None
        self.last = None
        self.index = torch.cuda.current_device()
        self.read = lambda: None
        try:
            import pynvml
            pynvml.nvmlInit()
            h = pynvml.nvmlDeviceGetHandleByIndex(self.index)
            self.read = lambda: float(pynvml.nvmlDeviceGetClockInfo(h, pynvml.NVML_CLOCK_SM))
            self.h = h
            return
        except Exception:
            pass
        try:
            import ctypes
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit_v2 failed")
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
                raise OSError("nvmlDeviceGetHandleByIndex_v2 failed")
            clk = ctypes.c_uint()

            def read():
                # NVML_CLOCK_SM = 1
                return float(clk.value) if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 else None

            self.read = read
            self.h = h
        except Exception as e:               # fall back to one nvidia-smi query per row
            sys.stderr.write("NVML unavailable (%s); row clocks from nvidia-smi\n" % e)
            self.h = None

    def query(self):
        """One nvidia-smi reading of the SM clock (MHz), or None."""
        try:
            out = subprocess.run(["nvidia-smi", "-i", str(self.index), "--query-gpu=clocks.sm",
                                  "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=10)
            return float(out.stdout.strip().splitlines()[0])
        except Exception:
            return None


_SM_CLOCK = None


def timed_reps(fn, reps, flush, stream, clocks=None):
    """Device times (ms) of `reps` runs of fn, each timed alone: the GPU is
    synchronised after every run (so each starts from an idle GPU at its
    burst clock) and L2 is flushed before it.  Between the flush and the
    run's first event the device sleeps ~0.2 ms, so the host has enqueued
    the run before the GPU reaches its events: a run's time never includes
    the host's time to launch it (which a busy host can stretch past the
    flush that would otherwise hide it)."""
    ts = []
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(reps):
        flush()
        torch.cuda._sleep(400_000)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
        if clocks is not None:
            clocks.append(_SM_CLOCK.read() if _SM_CLOCK is not None else None)
    return ts


def _time(fn, reps, warm, flush, stream):
    """Trimmed mean of `reps` event-timed runs, L2 flushed before each;
    records the median SM clock read right after each run in _SM_CLOCK.last."""
    global _SM_CLOCK
    if _SM_CLOCK is None:
        _SM_CLOCK = _SmClock()
    # a short idle first, so that a row does not start under the power cap
    # the rows before it drove the part into; then flushed runs for at least
    # 30 ms (and `warm` of them), so that clocks and the memory system are
    # back at full speed after the idle
    time.sleep(0.3)
    t0, n = time.time(), 0
    while n < warm or time.time() - t0 < 0.03:
        flush()
        fn()
        n += 1
        if n % 8 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    mhz = []
    ts = timed_reps(fn, reps, flush, stream, mhz)
    mhz = [c for c in mhz if c is not None]
    _SM_CLOCK.last = statistics.median(mhz) if mhz else _SM_CLOCK.query()
    return trimmed_mean(ts)


def trimmed_mean(ts, cut=0.2):
    """Mean of the middle 60% of the samples.  CUDA event times on this part
    come in steps of about 2 us, so the median of a ~20 us kernel sits on one
    step or the next; the mean of the middle samples averages the steps out
    while still dropping the outliers a median would."""
    v = sorted(ts)
    k = int(len(v) * cut)
    mid = v[k:len(v) - k] or v
    return sum(mid) / len(mid)


def _row_clock():
    return None if _SM_CLOCK is None else _SM_CLOCK.last


ROW_SECTIONS = ("dense", "wgrad", "moe_up", "moe_down", "swiglu")


def measure_rows(F, S, dev, flush, pk, sections=ROW_SECTIONS):
    """Each step of the path on its own workload, median of timed reps.
    `sections` picks which groups of rows run (each builds its own inputs)."""
    st = torch.cuda.current_stream()
    reps, warm = 20, 3
    fp8_peak = pk["bf16"] * 2.0
    out = {}

    def hbm_row(name, ms, nbytes, workload):
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = dict(workload=workload, ms=round(ms, 5), bound="hbm", achieved=round(gbs, 1), unit="GB/s",
                         algorithmic_bytes=int(nbytes), peak=pk["hbm"], frac=round(gbs / pk["hbm"], 4),
                         frac_of_nominal_8000=round(gbs / HBM_NOMINAL_GBS, 4), sm_mhz=_row_clock())

    def grouped_row(name, ms, flop, moved, wbytes, workload):
        """A grouped GEMM streams every expert's weights once: HBM-bound (AI ~
        2 x rows per expert FLOP/B, below the ridge), so the row's bound and
        fraction are HBM's; the tensor-peak fraction is kept beside them."""
        gbs = moved / (ms * 1e-3) / 1e9
        tf = flop / (ms * 1e-3) / 1e12
        out[name] = dict(workload=workload, ms=round(ms, 5), bound="hbm", achieved=round(gbs, 1), unit="GB/s",
                         algorithmic_bytes=int(moved), weight_bytes=int(wbytes), peak=pk["hbm"],
                         frac=round(gbs / pk["hbm"], 4), frac_of_nominal_8000=round(gbs / HBM_NOMINAL_GBS, 4),
                         tflops=round(tf, 1), tensor_frac=round(tf / fp8_peak, 4),
                         tensor_frac_of_nominal_4500=round(tf / FP8_NOMINAL_TFLOPS, 4), sm_mhz=_row_clock())

    def tensor_row(name, ms, flop, workload, extra=None):
        tf = flop / (ms * 1e-3) / 1e12
        r = dict(workload=workload, ms=round(ms, 5), bound="tensor", achieved=round(tf, 1), unit="TFLOP/s",
                 flop=flop, peak=round(fp8_peak, 1), frac=round(tf / fp8_peak, 4),
                 frac_of_nominal_4500=round(tf / FP8_NOMINAL_TFLOPS, 4), sm_mhz=_row_clock())
        if extra:
            r.update(extra)
        out[name] = r

    if "dense" in sections:
        measure_dense_rows(F, S, dev, flush, st, reps, warm, hbm_row, tensor_row, out)
    if "wgrad" in sections:
        measure_wgrad_rows(F, S, dev, flush, st, reps, warm, hbm_row, tensor_row, out)
    if "moe_up" in sections:
        measure_moe_up_rows(F, S, dev, flush, st, reps, warm, hbm_row, grouped_row, out)
    if "moe_down" in sections:
        measure_moe_down_rows(F, S, dev, flush, st, reps, warm, hbm_row, grouped_row, out)
    if "swiglu" in sections:
        measure_swiglu_rows(F, dev, flush, st, reps, warm, hbm_row)
    torch.cuda.synchronize()
    if F.fp8_get_status() != 0:
        raise RuntimeError("device status set while timing rows")
    return out


def measure_dense_rows(F, S, dev, flush, st, reps, warm, hbm_row, tensor_row, out):
    d = S.dense_linear()
    x, w = d["x"].to(dev), d["w"].to(dev)
    qx, sx = F.fp8_quant_act_1x128(x)
    qw, sw = F.fp8_quant_weight_128x128(w)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ms = _time(lambda: F.fp8_quant_act_1x128(x, qx, sx), reps, warm, flush, st)
    hbm_row("a1_quant_act_1x128", ms, M * K * 3 + M * (K // 128) * 4, "X [4096,7168]")
    ms = _time(lambda: F.fp8_quant_weight_128x128(w, qw, sw), reps, warm, flush, st)
    hbm_row("a3_quant_weight_128x128", ms, N * K * 3 + (N // 128) * (K // 128) * 4, "W [7168,7168]")
    ms_whole = _time(lambda: F.fp8_gemm_blockscaled(qx, sx, qw, sw, 0, torch.bfloat16, d=y, split=False),
                     reps, warm, flush, st)
    ms = _time(lambda: F.fp8_gemm_blockscaled(qx, sx, qw, sw, 0, torch.bfloat16, d=y), reps, warm, flush, st)
    tensor_row("a4_gemm_dense", ms, GEMM_FLOP, "4096x7168x7168 -> bf16",
               dict(unsplit_ms=round(ms_whole, 5)))
    # the same GEMM quantising D in its epilogue (1x128 tiles along N) for the next GEMM;
    # unfused, that is the bf16-out GEMM plus a 1x128 quantiser pass over a [4096,7168] bf16 tensor
    q8, s8 = F.fp8_gemm_blockscaled_q8(qx, sx, qw, sw)
    ms = _time(lambda: F.fp8_gemm_blockscaled_q8(qx, sx, qw, sw, 0, 0, q8, s8), reps, warm, flush, st)
    tensor_row("f2_gemm_dense_q8", ms, GEMM_FLOP, "4096x7168x7168 -> E4M3 + 1x128 scales (quantised in the epilogue)",
               dict(unfused_ms=round(out["a4_gemm_dense"]["ms"] + out["a1_quant_act_1x128"]["ms"], 5)))
    del q8, s8
    # Dgrad: dX = dY W from the transposed 128x128-block codes of W
    qwT, swT = F.fp8_transpose_128x128(qw, sw)
    ms = _time(lambda: F.fp8_transpose_128x128(qw, sw, qwT, swT), reps, warm, flush, st)
    hbm_row("a8_transpose_128x128", ms, 2 * N * K + 2 * (N // 128) * (K // 128) * 4, "W codes [7168,7168] -> W^T codes")
    dy = (torch.randn((M, N), generator=torch.Generator(device=dev).manual_seed(3), device=dev) * 1e-3).to(torch.bfloat16)
    qdy, sdy = F.fp8_quant_act_1x128(dy)
    ms = _time(lambda: F.fp8_gemm_blockscaled(qdy, sdy, qwT, swT, 0, torch.bfloat16, d=y), reps, warm, flush, st)
    tensor_row("a8_gemm_dgrad", ms, GEMM_FLOP, "dX = dY W, 4096x7168x7168 -> bf16")
    # power-of-two scales: the same GEMM with the scales applied by the tensor core
    P = F.FP8_SCALE_POW2
    qx2, sx2 = F.fp8_quant_act_1x128(x, flags=P)
    qw2, sw2 = F.fp8_quant_weight_128x128(w, flags=P)
    ms = _time(lambda: F.fp8_gemm_blockscaled_pow2(qx2, sx2, qw2, sw2, 0, torch.bfloat16, d=y), reps, warm, flush, st)
    tensor_row("f1_gemm_dense_pow2", ms, GEMM_FLOP, "4096x7168x7168 -> bf16, pow-2 scales as UE8M0 (microscaled MMA)")
    del x, w, qx, qw, y, qwT, dy, qdy, qx2, qw2


def measure_wgrad_rows(F, S, dev, flush, st, reps, warm, hbm_row, tensor_row, out):
    d = S.wgrad()
    T, H = d["dy"].shape
    dy, xx = d["dy"].to(dev), d["x"].to(dev)
    qa, sa = F.fp8_quant_act_128x1(dy)
    qb, sb = F.fp8_quant_act_128x1(xx)
    dw = torch.empty((H, H), dtype=torch.float32, device=dev)
    ms = _time(lambda: F.fp8_quant_act_128x1(dy, qa, sa), reps, warm, flush, st)
    hbm_row("a2_quant_act_128x1", ms, T * H * 3 + (T // 128) * H * 4, "dY [8192,7168] -> dY^T")
    ms = _time(lambda: F.fp8_gemm_blockscaled(qa, sa, qb, sb, F.FP8_BSCALE_ROW, torch.float32, d=dw),
               reps, warm, flush, st)
    tensor_row("a5_gemm_wgrad", ms, 2.0 * H * H * T, "dW = dY^T X, 7168x7168x8192 -> fp32")
    P = F.FP8_SCALE_POW2
    qa2, sa2 = F.fp8_quant_act_128x1(dy, flags=P)
    qb2, sb2 = F.fp8_quant_act_128x1(xx, flags=P)
    ms = _time(lambda: F.fp8_gemm_blockscaled_pow2(qa2, sa2, qb2, sb2, F.FP8_BSCALE_ROW, torch.float32, d=dw),
               reps, warm, flush, st)
    tensor_row("f1_gemm_wgrad_pow2", ms, 2.0 * H * H * T, "dW = dY^T X, 7168x7168x8192 -> fp32, pow-2 scales")
    del dy, xx, qa, qb, dw, qa2, qb2


def measure_moe_up_rows(F, S, dev, flush, st, reps, warm, hbm_row, grouped_row, out):
    E, k, K = 256, 8, 7168
    mu = S.moe_up(with_weights=False)
    x, logits = mu["x"].to(dev), mu["logits"].to(dev)
    Tn = x.shape[0]
    r = F.fp8_moe_route_topk(logits, k)
    ms = _time(lambda: F.fp8_moe_route_topk(logits, k, out=r), reps, warm, flush, st)
    out["a7_route_topk"] = dict(workload="logits [4096,256] -> top-8", ms=round(ms, 5), bound="latency")
    qx, sx = F.fp8_quant_act_1x128(x)
    qa, sa = F.fp8_permute_rows(qx, sx, r["src_row"])
    ms = _time(lambda: F.fp8_permute_rows(qx, sx, r["src_row"], qa, sa), reps, warm, flush, st)
    R = Tn * k
    hbm_row("a7_permute_rows", ms, 2 * R * (K + (K // 128) * 4) + R * 4, "[4096,7168] fp8 -> [32768,7168]")
    Nu = 4096
    wst = S.expert_weights(0, E, Nu, K, device=dev)
    qwu, swu = F.fp8_quant_weight_128x128(wst)
    ms = _time(lambda: F.fp8_quant_weight_128x128(wst, qwu, swu), 3, 1, flush, st)
    hbm_row("a3_quant_weight_moe_up", ms, E * Nu * K * 3 + E * (Nu // 128) * (K // 128) * 4, "256 x [4096,7168]")
    P = F.FP8_SCALE_POW2
    qwu2, swu2 = F.fp8_quant_weight_128x128(wst, flags=P)
    del wst
    yu = torch.empty((R, Nu), dtype=torch.bfloat16, device=dev)
    ms = _time(lambda: F.fp8_grouped_gemm_blockscaled(qa, sa, qwu, swu, r["off"], d=yu), reps, warm, flush, st)
    wbytes = E * Nu * K
    moved = wbytes + R * K + R * Nu * 2
    grouped_row("a6_grouped_moe_up", ms, 2.0 * R * Nu * K, moved, wbytes, "32768 rows, 256 experts, N=4096, K=7168")
    qx2, sx2 = F.fp8_quant_act_1x128(x, flags=P)
    qa2, sa2 = F.fp8_permute_rows(qx2, sx2, r["src_row"])
    ms = _time(lambda: F.fp8_grouped_gemm_blockscaled_pow2(qa2, sa2, qwu2, swu2, r["off"], d=yu), reps, warm, flush, st)
    grouped_row("f1_grouped_moe_up_pow2", ms, 2.0 * R * Nu * K, moved, wbytes,
                "32768 rows, 256 experts, N=4096, K=7168, pow-2 scales (microscaled MMA)")
    del qwu, qwu2, yu, qa, qx, qa2, qx2


def measure_moe_down_rows(F, S, dev, flush, st, reps, warm, hbm_row, grouped_row, out):
    E, k, P = 256, 8, F.FP8_SCALE_POW2
    md = S.moe_down(with_weights=False)
    h, logits = md["h"].to(dev), md["logits"].to(dev)
    r = F.fp8_moe_route_topk(logits, k)
    Kd, Nd = 2048, 7168
    Tn = logits.shape[0]
    R = Tn * k
    qh, sh = F.fp8_quant_act_1x128(h)
    ms = _time(lambda: F.fp8_quant_act_1x128(h, qh, sh), reps, warm, flush, st)
    hbm_row("a1_quant_act_1x128_moe_down", ms, R * Kd * 3 + R * (Kd // 128) * 4, "h [32768,2048]")
    wst = S.expert_weights(1, E, Nd, Kd, device=dev)
    qwd, swd = F.fp8_quant_weight_128x128(wst)
    qwd2, swd2 = F.fp8_quant_weight_128x128(wst, flags=P)
    del wst
    yd = torch.empty((R, Nd), dtype=torch.bfloat16, device=dev)
    ms = _time(lambda: F.fp8_grouped_gemm_blockscaled(qh, sh, qwd, swd, r["off"], d=yd), reps, warm, flush, st)
    wbytes = E * Nd * Kd
    moved = wbytes + R * Kd + R * Nd * 2
    grouped_row("a6_grouped_moe_down", ms, 2.0 * R * Nd * Kd, moved, wbytes, "32768 rows, 256 experts, N=7168, K=2048")
    qh2, sh2 = F.fp8_quant_act_1x128(h, flags=P)
    yd2 = torch.empty((R, Nd), dtype=torch.bfloat16, device=dev)
    ms = _time(lambda: F.fp8_grouped_gemm_blockscaled_pow2(qh2, sh2, qwd2, swd2, r["off"], d=yd2), reps, warm, flush, st)
    grouped_row("f1_grouped_moe_down_pow2", ms, 2.0 * R * Nd * Kd, moved, wbytes,
                "32768 rows, 256 experts, N=7168, K=2048, pow-2 scales (microscaled MMA)")
    del qwd2, qh2, yd2
    outc = torch.empty((Tn, Nd), dtype=torch.bfloat16, device=dev)
    ms = _time(lambda: F.fp8_moe_combine_bf16(yd, r["pos"], r["gate"], out=outc), reps, warm, flush, st)
    hbm_row("a7_combine_bf16", ms, R * Nd * 2 + Tn * Nd * 2 + R * 8, "[32768,7168] bf16 -> [4096,7168]")


def measure_swiglu_rows(F, dev, flush, st, reps, warm, hbm_row):
    """The MoE down-projection input formed from the up-projection output
    (32768 dispatched rows, gate | up of 2 x 2048): SwiGLU fused with
    power-of-two 1x128 quantisation."""
    R, Kd = 32768, 2048
    yup = torch.randn((R, 2 * Kd), generator=torch.Generator(device=dev).manual_seed(5), device=dev).to(torch.bfloat16)
    qg, sg = F.fp8_swiglu_quant_1x128(yup, Kd)
    ms = _time(lambda: F.fp8_swiglu_quant_1x128(yup, Kd, qg, sg), reps, warm, flush, st)
    hbm_row("f4_swiglu_quant_1x128_pow2", ms, R * 2 * Kd * 2 + R * Kd + R * (Kd // 128) * 4,
            "[32768, 2 x 2048] bf16 -> h = SiLU(gate)*up as E4M3 + pow-2 scales")


# ---------------------------------------------------------------- oracle (CPU) arm
def _dense_sample(S, oracle, d, rows):
    """1x128 quantisation of the first `rows` rows of X, 128x128 quantisation
    of all of W, and those rows of the GEMM in fp64: seconds, FLOP."""
    xb = S.bf16_bits(d["x"][:rows])
    wb = S.bf16_bits(d["w"])
    t0 = time.perf_counter()
    qa, sa = oracle.quant_act_1x128(xb)
    qb, sb = oracle.quant_weight_128x128(wb)
    oracle.gemm_blockscaled(qa, sa, qb, sb, 0)
    dt = time.perf_counter() - t0
    return dt, 2.0 * rows * wb.shape[0] * xb.shape[1]


def _rate(nbytes_or_flop, sec, unit):
    scale = 1e9 if unit in ("GB/s", "GFLOP/s") else 1e12
    return round(nbytes_or_flop / sec / scale, 4)


def cpu_baseline(S, d=None, dev=None):
    """The oracle, as it stands, on the host's cores (OpenMP, all threads), on
    a bounded sample of every workload (about 10-20 s of CPU work in all):
    quantisers, routing, dispatch and combine on the full tensors, GEMMs in
    fp64 on a stated fixed part of the rows.  `value` is the dense-linear
    step's sample (512 of 4096 rows with all of W) as GEMM TFLOP/s; `configs`
    has each workload's steps with their own rates."""
    import numpy as np
    import oracle
    oracle.build()
    cores = oracle.max_threads()
    T = time.perf_counter

    def step(fn, amount, unit, what):
        t0 = T()
        out = fn()
        dt = T() - t0
        return out, dict(seconds=round(dt, 3), value=_rate(amount, dt, unit), unit=unit, sample=what)

    cfgs = {}
    # tiny dense (everything in full)
    td = S.tiny_dense()
    xb, wb = S.bf16_bits(td["x"]), S.bf16_bits(td["w"])
    c = {}
    (qa, sa), c["quant_act_1x128"] = step(lambda: oracle.quant_act_1x128(xb), xb.size * 3, "GB/s", "X [128,512], all")
    (qb, sb), c["quant_weight_128x128"] = step(lambda: oracle.quant_weight_128x128(wb), wb.size * 3, "GB/s",
                                               "W [256,512], all")
    _, c["gemm_fp64"] = step(lambda: oracle.gemm_blockscaled(qa, sa, qb, sb, 0), 2.0 * 128 * 256 * 512, "GFLOP/s",
                             "128x256x512, all")
    cfgs["tiny_dense"] = c
    # dense linear: quantisers in full, GEMM on 512 of 4096 rows
    d = d or S.dense_linear()
    xb, wb = S.bf16_bits(d["x"]), S.bf16_bits(d["w"])
    c = {}
    (qa, sa), c["quant_act_1x128"] = step(lambda: oracle.quant_act_1x128(xb), xb.size * 3, "GB/s",
                                          "X [4096,7168], all")
    (qb, sb), c["quant_weight_128x128"] = step(lambda: oracle.quant_weight_128x128(wb), wb.size * 3, "GB/s",
                                               "W [7168,7168], all")
    rows = np.arange(512)
    _, c["gemm_fp64"] = step(lambda: oracle.gemm_blockscaled(qa, sa, qb, sb, 0, rows=rows), 2.0 * 512 * N * K,
                             "GFLOP/s", "rows 0..511 of 4096 x all 7168 columns, K 7168")
    cfgs["dense_linear"] = c
    head_dt, head_flop = _dense_sample(S, oracle, d, 512)
    del d, xb, wb, qa, qb
    # MoE up-projection: routing, quantisation and dispatch in full; 4 experts'
    # weights quantised; the grouped GEMM on the rows of 2 experts x all 4096 columns
    mu = S.moe_up(with_weights=False)
    c = {}
    r, c["route_topk"] = step(lambda: oracle.route_topk(mu["logits"].numpy(), 8), 4096 * 256 * 4, "GB/s",
                              "logits [4096,256] -> top-8, all")
    xb = S.bf16_bits(mu["x"])
    (qx, sx), c["quant_act_1x128"] = step(lambda: oracle.quant_act_1x128(xb), xb.size * 3, "GB/s",
                                          "X [4096,7168], all")
    (qa, sa), c["permute_rows"] = step(lambda: oracle.permute_rows(qx, sx, r["src_row"]), 2 * 32768 * (7168 + 224),
                                       "GB/s", "[4096,7168] -> [32768,7168], all")
    wdev = dev if dev is not None else "cpu"
    wq = {}
    wsample = [S.bf16_bits(S.expert_weight(0, e, 4096, 7168, device=wdev)) for e in range(4)]
    _, c["quant_weight_128x128"] = step(lambda: [wq.__setitem__(e, oracle.quant_weight_128x128(w))
                                                 for e, w in enumerate(wsample)],
                                        4 * 4096 * 7168 * 3, "GB/s", "experts 0..3 of 256, [4096,7168] each")
    off = r["off"]
    lo, hi = int(off[0]), int(off[2])
    _, c["grouped_gemm_fp64"] = step(
        lambda: [oracle.gemm_blockscaled(qa[off[e]:off[e + 1]], np.ascontiguousarray(sa[:, off[e]:off[e + 1]]),
                                         wq[e][0], wq[e][1], 0) for e in range(2)],
        2.0 * (hi - lo) * 4096 * 7168, "GFLOP/s", "experts 0, 1 (%d rows) x all 4096 columns, K 7168" % (hi - lo))
    cfgs["moe_up"] = c
    del mu, xb, qx, qa, wq, wsample
    # MoE down-projection: routing, quantisation and combine in full; 4
    # experts' weights; the grouped GEMM on the rows of 2 experts
    md = S.moe_down(with_weights=False)
    c = {}
    r, c["route_topk"] = step(lambda: oracle.route_topk(md["logits"].numpy(), 8), 4096 * 256 * 4, "GB/s",
                              "logits [4096,256] -> top-8, all")
    hb = S.bf16_bits(md["h"])
    (qh, sh), c["quant_act_1x128"] = step(lambda: oracle.quant_act_1x128(hb), hb.size * 3, "GB/s",
                                          "h [32768,2048], all")
    wq = {}
    wsample = [S.bf16_bits(S.expert_weight(1, e, 7168, 2048, device=wdev)) for e in range(4)]
    _, c["quant_weight_128x128"] = step(lambda: [wq.__setitem__(e, oracle.quant_weight_128x128(w))
                                                 for e, w in enumerate(wsample)],
                                        4 * 7168 * 2048 * 3, "GB/s", "experts 0..3 of 256, [7168,2048] each")
    off = r["off"]
    lo, hi = int(off[0]), int(off[2])
    _, c["grouped_gemm_fp64"] = step(
        lambda: [oracle.gemm_blockscaled(qh[off[e]:off[e + 1]], np.ascontiguousarray(sh[:, off[e]:off[e + 1]]),
                                         wq[e][0], wq[e][1], 0) for e in range(2)],
        2.0 * (hi - lo) * 7168 * 2048, "GFLOP/s", "experts 0, 1 (%d rows) x all 7168 columns, K 2048" % (hi - lo))
    yb = S.bf16_bits(torch.randn((32768, 7168), generator=torch.Generator().manual_seed(44)).to(torch.bfloat16))
    _, c["combine_bf16"] = step(lambda: oracle.moe_combine(yb, r["pos"], r["gate"]),
                                32768 * 7168 * 2 + 4096 * 7168 * 2, "GB/s",
                                "expert outputs [32768,7168] -> [4096,7168], all")
    cfgs["moe_down"] = c
    del md, hb, qh, wq, wsample, yb
    # Wgrad: both 128x1 quantisations in full; the GEMM on 64 of 7168 rows
    wg = S.wgrad()
    c = {}
    dyb, xb = S.bf16_bits(wg["dy"]), S.bf16_bits(wg["x"])
    (qa, sa), c["quant_act_128x1_dy"] = step(lambda: oracle.quant_act_128x1(dyb), dyb.size * 3, "GB/s",
                                             "dY [8192,7168] -> dY^T, all")
    (qb, sb), c["quant_act_128x1_x"] = step(lambda: oracle.quant_act_128x1(xb), xb.size * 3, "GB/s",
                                            "X [8192,7168] -> X^T, all")
    rows = np.arange(64)
    _, c["gemm_fp64"] = step(lambda: oracle.gemm_blockscaled(qa, sa, qb, sb, 1, rows=rows),
                             2.0 * 64 * 7168 * 8192, "GFLOP/s", "rows 0..63 of 7168 x all 7168 columns, K 8192")
    cfgs["wgrad"] = c
    total = sum(v["seconds"] for c in cfgs.values() for v in c.values()) + head_dt
    return {"value": round(head_flop / head_dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "seconds": round(head_dt, 2),
            "sample": "dense-linear step on 512 of 4096 rows: quantise those X rows (1x128) and all of W "
                      "(128x128), then those rows of the GEMM in fp64",
            "seconds_all_configs": round(total, 1), "configs": cfgs}


def run_reference(args, ws, rank):
    from fp8_fine_grained_16_b300 import synthetic as S
    if rank != 0:
        return None
    import oracle
    oracle.build()
    d = S.dense_linear()
    per = []
    rows = 32                       # per step: about 0.1-0.5 s of oracle work
    d_small = dict(x=d["x"][:rows], w=d["w"][:1024])
    for i in range(args.warmup + args.steps):
        dt, flop = _dense_sample(S, oracle, d_small, rows)
        if i >= args.warmup:
            per.append(dt)
    ms = 1e3 * sum(per) / len(per)
    v = round(flop / (ms * 1e-3) / 1e12, 6)
    cb = {"value": v, "unit": "TFLOP/s", "cores": oracle.max_threads(), "kind": "oracle",
          "sample": "each step: 1x128 quantisation of 32 of 4096 X rows, 128x128 quantisation of 1024 of 7168 W "
                    "rows, and that 32 x 1024 corner of the dense-linear GEMM in fp64"}
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
        "config": {"workload": WORKLOAD + " -- oracle on a 32-row x 1024-column corner per step",
                   "l2": "n/a (CPU)"},
        "cpu_baseline": cb,
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------- single-kernel cases (for ncu)
CASES = ("dense", "wgrad", "wgrad_small", "q8", "dgrad_transpose", "quant_1x128", "quant_1x128_h", "quant_128x1",
         "quant_act_weight",
         "quant_128x128",
         "grouped_up_small", "grouped_down_small", "grouped_down_small_pow2", "route", "permute", "combine", "swiglu",
         "pow2_dense", "pow2_wgrad_small")


def run_case(name: str, reps: int):
    """One kernel of the path on a bounded synthetic case, launched 1 + reps
    times (the first launch warms up; L2 is flushed before each timed one):
    what an ncu capture of that kernel runs (`-k <kernel> -s 1 -c 1`).  Random E4M3 codes (NaN codes excluded)
    and log-uniform scales stand in for quantised operands; the grouped
    cases keep the MoE shapes with 32 experts of ~128 rows (Poisson) so a
    full-metric capture holds about 1 GB."""
    from fp8_fine_grained_16_b300 import build
    build.build()
    from fp8_fine_grained_16_b300 import fp8bs as F
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(0)

    def codes(*shape):
        c = torch.randint(0, 256, shape, dtype=torch.uint8, device=dev, generator=g)
        c[(c & 0x7F) == 0x7F] = 0x3C
        return c

    def scales(*shape):
        return torch.exp(torch.empty(shape, device=dev).uniform_(-6.9, 1.38, generator=g))

    def bf16(*shape):
        return torch.randn(shape, device=dev, generator=g).to(torch.bfloat16)

    def offsets(E, mean=128):
        cnt = torch.poisson(torch.full((E,), float(mean), device=dev), generator=g).to(torch.int64)
        off = torch.zeros(E + 1, dtype=torch.int32, device=dev)
        off[1:] = torch.cumsum(cnt, 0).to(torch.int32)
        return off, int(off[-1])

    if name in ("dense", "q8", "pow2_dense"):
        a, b = codes(M, K), codes(N, K)
        sa, sb = scales(K // 128, M), scales(N // 128, K // 128)
        if name == "pow2_dense":
            sa, sb = torch.exp2(torch.round(torch.log2(sa))), torch.exp2(torch.round(torch.log2(sb)))
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            fn = lambda: F.fp8_gemm_blockscaled_pow2(a, sa, b, sb, 0, torch.bfloat16, d=y)
        elif name == "q8":
            q8, s8 = F.fp8_gemm_blockscaled_q8(a, sa, b, sb)
            fn = lambda: F.fp8_gemm_blockscaled_q8(a, sa, b, sb, 0, 0, q8, s8)
        else:
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            fn = lambda: F.fp8_gemm_blockscaled(a, sa, b, sb, 0, torch.bfloat16, d=y)
        work = "%dx%dx%d" % (M, N, K)
    elif name in ("wgrad", "wgrad_small", "pow2_wgrad_small"):
        H, T = (7168, 8192) if name == "wgrad" else (2048, 8192)
        a, b = codes(H, T), codes(H, T)
        sa, sb = scales(T // 128, H), scales(T // 128, H)
        dw = torch.empty((H, H), dtype=torch.float32, device=dev)
        if name == "pow2_wgrad_small":
            sa, sb = torch.exp2(torch.round(torch.log2(sa))), torch.exp2(torch.round(torch.log2(sb)))
            fn = lambda: F.fp8_gemm_blockscaled_pow2(a, sa, b, sb, F.FP8_BSCALE_ROW, torch.float32, d=dw)
        else:
            fn = lambda: F.fp8_gemm_blockscaled(a, sa, b, sb, F.FP8_BSCALE_ROW, torch.float32, d=dw)
        work = "%dx%dx%d, per-row B scales, fp32 out" % (H, H, T)
    elif name == "dgrad_transpose":
        q, sq = codes(N, K), scales(N // 128, K // 128)
        qT, sT = F.fp8_transpose_128x128(q, sq)
        fn = lambda: F.fp8_transpose_128x128(q, sq, qT, sT)
        work = "W codes [7168,7168] -> W^T codes"
    elif name == "quant_1x128":
        x = bf16(M, K)
        qx, sx = F.fp8_quant_act_1x128(x)
        fn = lambda: F.fp8_quant_act_1x128(x, qx, sx)
        work = "X [4096,7168]"
    elif name == "quant_act_weight":
        x, w = bf16(M, K), bf16(N, K)
        qx, sx, qw, sw = F.fp8_quant_act_weight(x, w)
        fn = lambda: F.fp8_quant_act_weight(x, w, qx, sx, qw, sw)
        work = "X [4096,7168] and W [7168,7168], one launch"
    elif name == "quant_1x128_h":
        x = bf16(32768, 2048)
        qx, sx = F.fp8_quant_act_1x128(x)
        fn = lambda: F.fp8_quant_act_1x128(x, qx, sx)
        work = "h [32768,2048]"
    elif name == "quant_128x1":
        x = bf16(8192, 7168)
        qT, sT = F.fp8_quant_act_128x1(x)
        fn = lambda: F.fp8_quant_act_128x1(x, qT, sT)
        work = "dY [8192,7168] -> dY^T"
    elif name == "quant_128x128":
        w = bf16(N, K)
        qw, sw = F.fp8_quant_weight_128x128(w)
        fn = lambda: F.fp8_quant_weight_128x128(w, qw, sw)
        work = "W [7168,7168]"
    elif name in ("grouped_up_small", "grouped_down_small", "grouped_down_small_pow2"):
        E = 32
        Ng, Kg = (4096, 7168) if name == "grouped_up_small" else (7168, 2048)
        off, R = offsets(E)
        a, sa = codes(R, Kg), scales(Kg // 128, R)
        b, sb = codes(E, Ng, Kg), scales(E, Ng // 128, Kg // 128)
        y = torch.empty((R, Ng), dtype=torch.bfloat16, device=dev)
        if name == "grouped_down_small_pow2":
            sa, sb = torch.exp2(torch.round(torch.log2(sa))), torch.exp2(torch.round(torch.log2(sb)))
            fn = lambda: F.fp8_grouped_gemm_blockscaled_pow2(a, sa, b, sb, off, d=y)
        else:
            fn = lambda: F.fp8_grouped_gemm_blockscaled(a, sa, b, sb, off, d=y)
        work = "%d rows, 32 experts, N=%d, K=%d" % (R, Ng, Kg)
    elif name == "route":
        logits = torch.randn((4096, 256), device=dev, generator=g)
        r = F.fp8_moe_route_topk(logits, 8)
        wk = torch.empty(max(1, F.fp8_moe_route_workspace_size(4096, 256) // 4), dtype=torch.int32, device=dev)
        fn = lambda: F.fp8_moe_route_topk(logits, 8, out=r, work=wk)
        work = "logits [4096,256] -> top-8, offsets, positions"
    elif name in ("permute", "combine"):
        logits = torch.randn((4096, 256), device=dev, generator=g)
        r = F.fp8_moe_route_topk(logits, 8)
        if name == "permute":
            q, sq = codes(4096, 7168), scales(56, 4096)
            qo, so = F.fp8_permute_rows(q, sq, r["src_row"])
            fn = lambda: F.fp8_permute_rows(q, sq, r["src_row"], qo, so)
            work = "[4096,7168] fp8 -> [32768,7168] by top-8 of 256"
        else:
            y = bf16(32768, 7168)
            out = F.fp8_moe_combine_bf16(y, r["pos"], r["gate"])
            fn = lambda: F.fp8_moe_combine_bf16(y, r["pos"], r["gate"], out=out)
            work = "[32768,7168] bf16 -> [4096,7168]"
    elif name == "swiglu":
        yup = bf16(32768, 4096)
        qg, sg = F.fp8_swiglu_quant_1x128(yup, 2048)
        fn = lambda: F.fp8_swiglu_quant_1x128(yup, 2048, qg, sg)
        work = "[32768, 2 x 2048] bf16"
    else:
        raise SystemExit("unknown case %r (one of %s)" % (name, ", ".join(CASES)))
    st = torch.cuda.current_stream()
    flush = L2Flush(dev)
    fn()
    torch.cuda.synchronize()
    ts = timed_reps(fn, reps, flush, st)
    status = F.fp8_get_status()
    print(json.dumps({"case": name, "workload": work, "launches": 1 + reps, "ms_min": round(min(ts), 5),
                      "ms_median": round(statistics.median(ts), 5), "ms_trimmed_mean": round(trimmed_mean(ts), 5),
                      "status": status}))
    if status != 0:
        raise SystemExit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--rows", default="all",
                    help="all | none | comma-separated sections of %s" % ",".join(ROW_SECTIONS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", choices=CASES,
                    help="run one kernel on a bounded synthetic case (1 + --reps launches) and exit")
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args()
    if args.case:
        run_case(args.case, args.reps)
        return
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = dist_env()
    if args.impl == "reference":
        out = run_reference(args, ws, rank)
        if out is not None:
            print(json.dumps(out))
        return
    if ws > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    out = run_ours(args, ws, rank, local)
    if rank == 0:
        print(json.dumps(out))
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
