"""Throughput of the exact attention forward on B300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline] [--no-extra]
                    [--op forward|backward|decode]

A step is one attention forward over the whole workload (default: bf16,
causal, B=2, H=32, N=8192, D=128).  ``value`` is device-timed TFLOP/s with
inputs resident in HBM: the K steps are captured into one CUDA graph and its
replay is timed with CUDA events on the launching stream (the inputs, 403 MB,
exceed the 126 MB L2, so no flush is needed; workloads that fit in L2 are
timed launch by launch with a 256 MB buffer written before each).  The step is
one kernel, so ``roofline.achieved`` is that kernel's rate over the same time.
``e2e`` is the same metric through the C-ABI call on pinned host buffers
(``attn_fwd_host``): every step copies Q, K, V host->device and O, LSE
device->host inside the timed region, chunk by chunk, overlapped with the
kernels.  ``workloads`` carries the other forward workloads, the backward on
the headline shape and a KV-cache decode, each timed the same way with its
own clocks and roofline.  Under torchrun each rank runs its own replica of the
workload (weak scaling); the slowest rank's time is used.

``cpu_baseline`` (and ``--impl reference``) times the fp64 CPU oracle on the
host cores, whole planes at a time, one spawned process per core, on a
bounded sample of the same workload (rank 0 only).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from exact_io_aware_107_b300 import workloads as W  # noqa: E402

METRIC = "attention fwd TFLOPS (bf16, causal) and % of B300 dense bf16 tensor peak"
KERNEL_SOURCES = ["exact_io_aware_107_b300/csrc/fwd_bf16_sm103.cuh",
                  "exact_io_aware_107_b300/csrc/ptx.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, p), "rb").read())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("bf16_tflops", 1800.0), d.get("hbm_gbs", 6400.0), "measured"
    return 1800.0, 6400.0, "fallback"


def measured_traffic(workload: str):
    """DRAM bytes per launch from an ncu capture, if taken on the current kernel source."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    d = json.load(open(TRAFFIC_FILE))
    e = d.get(workload)
    if not e or e.get("kernel_source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """SM clocks and throttle reasons sampled during a timed region.

    NVML is polled every millisecond from a background thread (the timed
    regions are tens of milliseconds long); if NVML is unavailable,
    ``nvidia-smi -lms 10`` is used instead.
    """

    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap"}

    def __init__(self, local_index: int):
        cvd = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [t.strip() for t in cvd.split(",") if t.strip()]
        self.gpu = int(ids[local_index]) if local_index < len(ids) and ids[local_index].isdigit() \
            else local_index
        self.samples = []       # (sm_mhz, max_mhz, reason_bits)
        self._stop = threading.Event()
        self._thread = None
        self._proc = None
        self.source = None

    def _poll_nvml(self, nv, h):
        get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        mx = nv.nvmlDeviceGetMaxClockInfo(h, nv.NVML_CLOCK_SM)
        while not self._stop.is_set():
            try:
                self.samples.append((nv.nvmlDeviceGetClockInfo(h, nv.NVML_CLOCK_SM), mx,
                                     int(get_reasons(h))))
            except Exception:  # noqa: BLE001 - a failed query only loses one sample
                pass
            time.sleep(0.001)

    def _read_smi(self):
        for line in self._proc.stdout:
            f = [x.strip() for x in line.split(",")]
            try:
                bits = 0
                for bit, val in zip((0x8, 0x40, 0x20, 0x4), f[2:6]):
                    bits |= bit if val.lower() == "active" else 0
                self.samples.append((float(f[0]), float(f[1]), bits))
            except (ValueError, IndexError):
                continue

    def __enter__(self):
        try:
            import pynvml as nv
            nv.nvmlInit()
            h = nv.nvmlDeviceGetHandleByIndex(self.gpu)
            self._thread = threading.Thread(target=self._poll_nvml, args=(nv, h), daemon=True)
            self.source = "nvml"
        except Exception:  # noqa: BLE001 - fall back to the command-line tool
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", f"--id={self.gpu}",
                     "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                     "clocks_event_reasons.hw_thermal_slowdown,"
                     "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                     "--format=csv,noheader,nounits", "-lms", "10"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self._thread = threading.Thread(target=self._read_smi, daemon=True)
                self.source = "nvidia-smi"
                time.sleep(1.0)       # let the tool start before the timed region
            except OSError:
                self._thread = None
        if self._thread is not None:
            self._thread.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=5)
        return False

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "source": self.source}
        reasons = sorted({name for _, _, bits in self.samples
                          for bit, name in self.REASONS.items() if bits & bit})
        return {"sm_mhz": statistics.median(s[0] for s in self.samples),
                "sm_max_mhz": max(s[1] for s in self.samples), "reasons": reasons,
                "samples": len(self.samples), "source": self.source}


def system_info(dev) -> dict:
    """The device and software the line was measured on."""
    import torch
    prop = torch.cuda.get_device_properties(dev)
    info = {"sms": prop.multi_processor_count, "cc": f"{prop.major}.{prop.minor}",
            "torch": torch.__version__, "cuda_runtime": torch.version.cuda,
            "host_cores": host_cores(), "cgroup_cpu_limit": cgroup_cpu_limit()}
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader",
                              "-i", str(torch.cuda.current_device())],
                             capture_output=True, text=True, timeout=20).stdout.strip()
        info["driver"] = out.splitlines()[0] if out else None
    except (OSError, subprocess.SubprocessError):
        info["driver"] = None
    try:
        from exact_io_aware_107_b300 import _binding
        info["library_version"] = int(_binding.attn_version())
    except Exception:  # noqa: BLE001 - informational only
        info["library_version"] = None
    return info


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# CPU oracle timing (the cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def cgroup_cpu_limit():
    """CPUs' worth of time the cgroup quota allows this process (None: no quota)."""
    try:
        quota, period = open("/sys/fs/cgroup/cpu.max").read().split()[:2]
        if quota != "max" and int(period) > 0:
            return max(1, -(-int(quota) // int(period)))
    except (OSError, ValueError):
        pass
    try:
        quota = int(open("/sys/fs/cgroup/cpu/cpu.cfs_quota_us").read())
        period = int(open("/sys/fs/cgroup/cpu/cpu.cfs_period_us").read())
        if quota > 0 and period > 0:
            return max(1, -(-quota // period))
    except (OSError, ValueError):
        pass
    return None


def host_cores() -> int:
    """Cores this process may run on: the affinity mask, capped by a cgroup CPU quota."""
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    q = cgroup_cpu_limit()
    return min(n, q) if q else n


def _blas_single_thread():
    """One BLAS thread in this process inside the block (the oracle's helper)."""
    from oracle.threads import blas_threads
    return blas_threads(1)


# The oracle is timed in the form the parity tests run it: oracle.attention_plane
# on whole planes (the full score matrix up to 4096 rows, 512-row slabs above),
# one plane per task.  A unit of work is one plane, or its last UNIT_ROWS query
# rows when it is longer (those rows see the most keys under the causal mask).
UNIT_ROWS = 8192


def _oracle_units(w, x):
    """(q_rows, k, v) fp32 arrays per unit of the workload, in plane order.

    The fp32 arrays are exact images of the 16-bit inputs; the worker widens
    them to fp64 (also exactly) before calling the oracle."""
    def f32(t):
        import torch
        return t.detach().to(torch.float32).numpy()
    units = []
    if w.varlen is None:
        for b in range(w.B):
            for h in range(w.H):
                units.append((x["q"][b, h], x["k"][b, h], x["v"][b, h]))
    else:
        cu = x["cu_seqlens"]
        cuk = x["cu_seqlens_k"] if x["cu_seqlens_k"] is not None else cu
        for s in range(len(cu) - 1):
            for h in range(w.H):
                units.append((x["q"][h, cu[s]:cu[s + 1]], x["k"][h, cuk[s]:cuk[s + 1]],
                              x["v"][h, cuk[s]:cuk[s + 1]]))
    out = []
    for q, k, v in units:
        r0 = max(0, q.shape[0] - UNIT_ROWS)
        out.append((f32(q[r0:]), f32(k), f32(v)))
    return out


def _unit_flops(q, k, causal, D) -> float:
    """FLOPs of one unit: 4 D per allowed (query, key) pair, the queries being
    the last rows of the plane (key j allowed for query i when j <= i + Nk - Nq)."""
    nq, nk = q.shape[0], k.shape[0]
    if not causal:
        return 4.0 * D * nq * nk
    i = np.arange(nq)
    return 4.0 * D * float(np.clip(i + 1 + (nk - nq), 0, nk).sum())


def _oracle_unit(job):
    """Worker: the oracle on one unit; returns its seconds in the worker."""
    import oracle
    q, k, v, scale, causal = job
    t0 = time.perf_counter()
    oracle.attention_plane(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64),
                           scale, causal)
    return time.perf_counter() - t0


def _oracle_worker_init():
    from oracle.threads import set_blas_threads
    set_blas_threads(1)


class OraclePool:
    """The oracle on whole planes, one plane per task, over `procs` spawned
    processes with one BLAS thread each.  Spawned, not forked: a process forked
    after CUDA has been initialised can hang.  procs == 1 runs in this process."""

    def __init__(self, w, units, procs: int):
        self.w, self.units, self.procs, self.ex = w, units, procs, None
        self.next = 0
        if procs > 1:
            import multiprocessing as mp
            from concurrent.futures import ProcessPoolExecutor
            from oracle.threads import single_thread_children
            # the workers read OPENBLAS_NUM_THREADS=1 (and its OpenMP/MKL
            # equivalents) when their BLAS loads; the initialiser sets it again
            with single_thread_children():
                self.ex = ProcessPoolExecutor(max_workers=procs,
                                              mp_context=mp.get_context("spawn"),
                                              initializer=_oracle_worker_init)
                # start every worker (and its imports) before anything is timed
                tiny = (np.zeros((4, w.D), np.float32),) * 3
                try:
                    list(self.ex.map(_oracle_unit, [tiny + (w.scale, w.causal)] * (2 * procs),
                                     timeout=300))
                except Exception:  # noqa: BLE001 - any failure: measure in-process instead
                    self.ex.shutdown(wait=False, cancel_futures=True)
                    self.ex, self.procs = None, 1

    def round(self):
        """One round: the next `procs` units (cycling over the workload), one per
        process.  Returns (flops, wall seconds, units)."""
        idx = [(self.next + i) % len(self.units) for i in range(self.procs)]
        self.next = (self.next + self.procs) % len(self.units)
        jobs = [self.units[i] + (self.w.scale, self.w.causal) for i in idx]
        flops = sum(_unit_flops(j[0], j[1], self.w.causal, self.w.D) for j in jobs)
        t0 = time.perf_counter()
        if self.ex is None:
            with _blas_single_thread():
                for j in jobs:
                    _oracle_unit(j)
        else:
            list(self.ex.map(_oracle_unit, jobs, timeout=1800))
        return flops, time.perf_counter() - t0, len(jobs)

    def close(self):
        if self.ex is not None:
            self.ex.shutdown()


def _unit_desc(w):
    return (f"whole planes (the last {UNIT_ROWS} query rows of longer ones)" if w.varlen is None
            else f"whole (sequence, head) planes (the last {UNIT_ROWS} rows of longer ones)")


def cpu_baseline(w, x, cpu_seconds: float = 20.0):
    """Oracle throughput on a bounded sample: rounds of one plane per process,
    one process per core, until about `cpu_seconds` of CPU work; if that is
    slower than one process (a host whose cores are shared or throttled), one
    process on the same kind of sample."""
    units = _oracle_units(w, x)
    procs = host_cores()
    one = OraclePool(w, units, 1)
    f1, dt1, _ = one.round()
    v1 = f1 / dt1 / 1e12
    pool = OraclePool(w, units, procs)
    flops = secs = 0.0
    n = 0
    try:
        while secs * pool.procs < cpu_seconds or n == 0:
            f, dt, k = pool.round()
            flops, secs, n = flops + f, secs + dt, n + k
    finally:
        pool.close()
    value, used = flops / secs / 1e12, pool.procs
    how = f"one plane per process, {used} processes"
    if used > 1 and value < v1:
        flops, secs, n = f1, dt1, 1
        while secs < cpu_seconds:
            f, dt, k = one.round()
            flops, secs, n = flops + f, secs + dt, n + k
        how = (f"one process ({used} processes ran at {value:.2e} TFLOP/s, below one process: "
               f"the host's cores are shared or throttled)")
        value, used = flops / secs / 1e12, 1
    return {"value": value, "unit": "TFLOP/s", "cores": used, "kind": "oracle",
            "value_1core": v1,
            "sample": f"fp64 oracle.attention_plane on {n} {_unit_desc(w)} of {w.name}, "
                      f"{how}, {secs:.1f} s wall; FLOPs counted as 4 D per allowed "
                      f"(query, key) pair; value_1core: one plane in one process "
                      f"({dt1:.2f} s)"}


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    x = W.generate(w)
    units = _oracle_units(w, x)
    pool = OraclePool(w, units, host_cores())
    try:
        # a process per core, unless that is slower than one process on this host
        if pool.procs > 1:
            one = OraclePool(w, units, 1)
            f1, t1, _ = one.round()
            fp, tp, _ = pool.round()
            if fp / tp < f1 / t1:
                pool.close()
                pool = one
        for _ in range(args.warmup):
            pool.round()
        flops = secs = 0.0
        n = 0
        for _ in range(args.steps):
            f, dt, k = pool.round()
            flops, secs, n = flops + f, secs + dt, n + k
    finally:
        pool.close()
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": pool.procs, "kind": "oracle",
                         "sample": f"each step: fp64 oracle.attention_plane on {pool.procs} "
                                   f"{_unit_desc(w)} of {w.name}, one per process "
                                   f"({n} units in the timed steps)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def workload_config(w):
    cfg = {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D, "causal": w.causal,
           "dtype_in": w.dtype, "flops_per_step": w.flops(),
           "l2": "inputs larger than L2 (no flush)" if 3 * w.hbm_bytes() / 4 > 126e6
           else "L2 flushed between steps"}
    if w.is_cross:
        cfg["Nk"] = w.n_keys
        cfg["mask_alignment"] = "bottom-right (key j allowed for query i when j <= i + Nk - N)"
    if w.varlen is not None:
        cfg["seq_lens"] = list(w.varlen)
    return cfg


# ---------------------------------------------------------------------------
# CUDA path
# ---------------------------------------------------------------------------

def graph_step_ms(step, steps, stream, dev, reps=1):
    """Milliseconds per step of `steps` calls of step(stream) captured into one
    CUDA graph and replayed (the same kernels back to back, without host
    launch gaps); the median over `reps` replays; None when the capture is
    refused."""
    g = capture_graph(step, steps, stream, dev)
    if g is None:
        return None
    import torch
    times = []
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / steps)
    return statistics.median(times)


def capture_graph(step, steps, stream, dev):
    """`steps` calls of step(st) captured into one CUDA graph (replayed once to
    check it), or None when the capture is refused."""
    import torch
    try:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.graph(g, stream=cap):
            for _ in range(steps):
                step(torch.cuda.current_stream(dev))
        stream.wait_stream(cap)
        g.replay()
        torch.cuda.synchronize()
        return g
    except Exception as e:  # noqa: BLE001 - the caller falls back to eager timing
        print(f"[bench] graph capture failed ({e})", file=sys.stderr)
        return None


def fits_in_l2(nbytes: float) -> bool:
    """Inputs that (mostly) fit in the 126 MB L2 are flushed between launches."""
    return nbytes <= 126e6


def time_steps(call, steps, warmup, stream, dev, local, ws, flush_needed):
    """Device time of `steps` calls of call(stream).

    Inputs larger than L2: the K calls are captured into one CUDA graph and
    its replay is timed with CUDA events on the launching stream (the kernels
    back to back, without host launch gaps).  Inputs that fit in L2: a 256 MB
    buffer is written before every call and each call's own events give its
    time; the same K calls warm in L2 (one graph) are timed beside.
    Returns (ms per step, how it was timed, clock summary, warm ms or None).
    """
    import torch
    from exact_io_aware_107_b300 import device_error
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flush_needed else None
    for _ in range(warmup):
        if flush is not None:
            flush.zero_()
        call(stream)
    torch.cuda.synchronize()
    if device_error() != 0:
        raise RuntimeError("device error during warm-up")
    graph = capture_graph(call, steps, stream, dev) if flush is None else None
    barrier(ws)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            if graph is not None:
                starts[0].record(stream)
                graph.replay()
                ends[0].record(stream)
            else:
                for i in range(steps):
                    if flush is not None:
                        flush.zero_()
                    starts[i].record(stream)
                    call(stream)
                    ends[i].record(stream)
        torch.cuda.synchronize()
    barrier(ws)
    if device_error() != 0:
        raise RuntimeError("device error in the timed region")
    warm = None
    if graph is not None:
        ms, how = starts[0].elapsed_time(ends[0]) / steps, "one CUDA graph of the K steps"
    else:
        ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / steps
        how = "per-launch CUDA events (graph capture refused)"
        if flush is not None:
            # Per-launch events can include host time: the GPU may reach the
            # start event before the call has been enqueued.  One graph of the
            # K (flush, call) pairs minus one graph of the K flushes alone gives
            # the calls' device time after a flush, with no host in between.
            both = graph_step_ms(lambda st: (flush.zero_(), call(st)), steps, stream, dev,
                                 reps=3)
            alone = graph_step_ms(lambda st: flush.zero_(), steps, stream, dev, reps=3)
            if both is not None and alone is not None and both > alone:
                ms = both - alone
                how = ("L2 flushed (256 MB written) before each launch: one CUDA graph of the "
                       "K (flush, launch) pairs minus one graph of the K flushes")
            else:
                how = "per-launch CUDA events, L2 flushed (256 MB written) before each launch"
            warm = graph_step_ms(call, steps, stream, dev)
    return ms, how, clk.summary(), warm


def device_inputs(x, dev):
    import torch
    q, k, v = (t.to(dev) for t in (x["q"], x["k"], x["v"]))
    cu = None if x["cu_seqlens"] is None else torch.as_tensor(x["cu_seqlens"]).to(dev)
    cuk = None if x["cu_seqlens_k"] is None else torch.as_tensor(x["cu_seqlens_k"]).to(dev)
    return q, k, v, cu, cuk


def forward_call(w, q, k, v, cu, cuk):
    """call(stream): one forward of the workload into fixed output buffers."""
    import torch
    from exact_io_aware_107_b300 import attention_forward
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)

    def call(st):
        attention_forward(q, k, v, causal=w.causal, scale=w.scale, cu_seqlens=cu, out=o, lse=lse,
                          stream=st, cu_seqlens_k=cuk)
    return call, o, lse


def tensor_peak():
    peak_tf, _, kind = load_peaks()
    src = (f"{kind} cuBLAS bf16 burst (MEASURED_PEAKS.json)" if kind == "measured"
           else "fallback 1.8 PFLOP/s")
    return peak_tf, src


def measure_forward(w, x, steps, warmup, dev, stream, local=0, ws=1):
    q, k, v, cu, cuk = device_inputs(x, dev)
    call, _, _ = forward_call(w, q, k, v, cu, cuk)
    ms, how, clocks, warm = time_steps(call, steps, warmup, stream, dev, local, ws,
                                       fits_in_l2(3 * w.hbm_bytes() / 4))
    return ms, how, clocks, warm


def measure_backward(w, x, steps, warmup, dev, stream, local=0):
    """Device ms per backward (prep, main and dQ kernels) of workload w."""
    import torch
    from exact_io_aware_107_b300 import _binding, attention_backward, attention_forward
    q, k, v, cu, cuk = device_inputs(x, dev)
    rng = np.random.default_rng(1)
    do = torch.from_numpy(rng.standard_normal(tuple(q.shape), dtype=np.float32)).to(q.dtype).to(dev)
    o, lse = attention_forward(q, k, v, causal=w.causal, scale=w.scale, cu_seqlens=cu,
                               cu_seqlens_k=cuk, stream=stream)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    rc, nbytes = _binding.attn_bwd_workspace_bytes(w.B, w.H, w.N, w.D, cu is not None)
    assert rc == 0
    wsb = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)

    def call(st):
        attention_backward(q, k, v, o, lse, do, causal=w.causal, scale=w.scale, cu_seqlens=cu,
                           cu_seqlens_k=cuk, dq=dq, dk=dk, dv=dv, workspace=wsb, stream=st)
    return time_steps(call, steps, warmup, stream, dev, local, 1,
                      fits_in_l2(5 * w.hbm_bytes() / 4))


def decode_bytes(B, H, Nq, Nk, D) -> float:
    """Algorithmic HBM bytes of one decode: K and V read once, Q read, O and LSE written."""
    return 2.0 * B * H * Nk * D * 2 + 2.0 * B * H * Nq * D * 2 + B * H * Nq * 4


def measure_decode(shape, steps, warmup, dev, stream, local=0):
    import torch
    from exact_io_aware_107_b300 import _binding, attention_decode
    B, H, Nq, Nk, D = shape
    rng = np.random.default_rng(0)

    def draw(*sh):
        return torch.from_numpy(rng.standard_normal(sh, dtype=np.float32)).to(torch.bfloat16)
    q, k, v = (t.to(dev) for t in (draw(B, H, Nq, D), draw(B, H, Nk, D), draw(B, H, Nk, D)))
    rc, nbytes = _binding.attn_decode_workspace_bytes(B, H, Nq, Nk, D)
    assert rc == 0
    wsb = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)

    def call(st):
        attention_decode(q, k, v, workspace=wsb, out=o, lse=lse, stream=st)
    ms, how, clocks, _ = time_steps(call, steps, warmup, stream, dev, local, 1,
                                    fits_in_l2(2 * B * H * Nk * D * 2))
    return ms, how, clocks, nbytes


_READ_GBS = {}


def hbm_read_gbs(dev, stream):
    """Read-only HBM bandwidth of this GPU (best of 5 streams over 4 GiB, far
    larger than L2), through the library's read probe; cached per device."""
    import torch
    from exact_io_aware_107_b300 import _binding
    key = str(dev)
    if key not in _READ_GBS:
        nbytes = 4 << 30
        buf = torch.ones(nbytes // 4, dtype=torch.int32, device=dev)
        out = torch.zeros(1, dtype=torch.int32, device=dev)
        best = float("inf")
        for i in range(6):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            rc = _binding.attn_hbm_read_probe(buf.data_ptr(), nbytes, out.data_ptr(),
                                              stream.cuda_stream)
            e1.record(stream)
            assert rc == 0
            torch.cuda.synchronize()
            if i > 0:
                best = min(best, e0.elapsed_time(e1))
        _READ_GBS[key] = nbytes / (best * 1e-3) / 1e9
        del buf
    return _READ_GBS[key]


def hbm_peak(dev, stream):
    """The larger of the measured copy bandwidth and this GPU's read-only stream."""
    _, copy_gbs, kind = load_peaks()
    read = hbm_read_gbs(dev, stream)
    return max(copy_gbs, read), {"copy_gbs": copy_gbs, "copy_source": f"{kind} (MEASURED_PEAKS.json)"
                                 if kind == "measured" else "fallback", "read_gbs": read,
                                 "read_source": "attn_hbm_read_probe over 4 GiB, best of 5, "
                                                "this GPU, this run"}


# The other workloads carried in the default line (the headline stays the
# causal N=8192 D=128 forward): the D=64 non-causal forward (L2-flushed and
# warm), the long peaked causal forward, the packed variable-length forward,
# the backward on the headline shape and a KV-cache decode.
EXTRA_FORWARD = ("bf16_b4_h16_n2048_d64", "bf16_causal_b1_h16_n32768_d128_peaked",
                 "bf16_varlen_causal_h32_d128")
EXTRA_DECODE = (8, 32, 1, 32768, 128)


def extra_workloads(args, dev, stream, local):
    import torch
    peak_tf, _ = tensor_peak()
    out = {}

    def fwd_entry(w, ms, how, clocks, warm):
        tf = w.flops() / (ms * 1e-3) / 1e12
        e = {"value": tf, "unit": "TFLOP/s", "ms_per_step": ms, "timing": how,
             "roofline": {"bound": "tensor", "achieved": tf, "peak": peak_tf,
                          "unit": "TFLOP/s", "frac": tf / peak_tf},
             "clocks": clocks, "flops_per_step": w.flops()}
        if warm is not None:
            wt = w.flops() / (warm * 1e-3) / 1e12
            e["warm_l2"] = {"value": wt, "unit": "TFLOP/s", "ms_per_step": warm,
                            "frac": wt / peak_tf, "timing": "one CUDA graph of the K steps, "
                                                            "inputs in L2"}
        return e

    for name in EXTRA_FORWARD:
        w = W.WORKLOADS[name]
        x = W.generate(w)
        ms, how, clocks, warm = measure_forward(w, x, args.steps, args.warmup, dev, stream, local)
        out[name] = fwd_entry(w, ms, how, clocks, warm)
        del x
        torch.cuda.empty_cache()
    w = W.WORKLOADS[W.HEADLINE]
    x = W.generate(w)
    ms, how, clocks, _ = measure_backward(w, x, args.steps, args.warmup, dev, stream, local)
    tf = 2.5 * w.flops() / (ms * 1e-3) / 1e12
    out["backward_" + w.name] = {
        "value": tf, "unit": "TFLOP/s (2.5x the forward's FLOPs)", "ms_per_step": ms,
        "timing": how, "roofline": {"bound": "tensor", "achieved": tf, "peak": peak_tf,
                                    "unit": "TFLOP/s", "frac": tf / peak_tf},
        "clocks": clocks, "kernels": "attn_bwd_prep_kernel, attn_bwd_bf16_kernel<128>, "
                                      "attn_bwd_dq_kernel"}
    del x
    torch.cuda.empty_cache()
    B, H, Nq, Nk, D = EXTRA_DECODE
    ms, how, clocks, _ = measure_decode(EXTRA_DECODE, args.steps, args.warmup, dev, stream, local)
    nb = decode_bytes(B, H, Nq, Nk, D)
    gbs = nb / (ms * 1e-3) / 1e9
    peak, src = hbm_peak(dev, stream)
    out[f"decode_b{B}_h{H}_nq{Nq}_nk{Nk}_d{D}"] = {
        "value": gbs, "unit": "GB/s", "ms_per_step": ms, "timing": how,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                     "frac": gbs / peak, "peak_source": src, "algorithmic_bytes": nb},
        "clocks": clocks}
    torch.cuda.empty_cache()
    return out


def run_ours(args, w):
    import torch
    from exact_io_aware_107_b300 import _binding, attention_forward, device_error

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    _binding.load()
    x = W.generate(w)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)

    # --- device-timed region (inputs resident) ---
    step_ms, timing, clocks, warm_ms = measure_forward(w, x, args.steps, args.warmup, dev, stream,
                                                       local, ws)
    ms_step = max_over_ranks(step_ms, ws)
    flops = w.flops()
    value = ws * flops / (ms_step * 1e-3) / 1e12
    # the dominant (and only) kernel of a step: its time per launch is the
    # step's own device time on this rank
    achieved = flops / (step_ms * 1e-3) / 1e12
    torch.cuda.empty_cache()

    # --- end-to-end region: pinned host buffers, copies inside the timed region ---
    q, k, v, cu, cuk = device_inputs(x, dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=dev)
    hq, hk, hv = (t.pin_memory() for t in (x["q"], x["k"], x["v"]))
    ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    e_steps = max(3, min(args.steps, 10))
    host_api = w.varlen is None and not w.is_cross
    if host_api:
        # the C-ABI call on host buffers: chunked copies in, kernels, copies back, overlapped
        from exact_io_aware_107_b300 import attention_forward_host
        kind = {"bf16": _binding.ATTN_BF16, "f16": _binding.ATTN_F16, "f32": _binding.ATTN_F32}
        rc, nb = _binding.attn_fwd_host_workspace_bytes(w.B, w.H, w.N, w.D, kind[w.dtype])
        assert rc == 0
        hws = torch.empty(max(nb, 256), dtype=torch.uint8, device=dev)

        def e2e_step():
            attention_forward_host(hq, hk, hv, causal=w.causal, scale=w.scale, out=ho, lse=hl,
                                   workspace=hws, stream=stream, non_blocking=True)
    else:
        def e2e_step():
            q.copy_(hq, non_blocking=True)
            k.copy_(hk, non_blocking=True)
            v.copy_(hv, non_blocking=True)
            attention_forward(q, k, v, causal=w.causal, scale=w.scale, cu_seqlens=cu, out=o,
                              lse=lse, stream=stream, cu_seqlens_k=cuk)
            ho.copy_(o, non_blocking=True)
            hl.copy_(lse, non_blocking=True)
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(ws)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    if device_error() != 0:
        raise RuntimeError("device error in the end-to-end region")
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e_steps, ws)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
    del q, k, v, o, lse
    torch.cuda.empty_cache()

    peak_tf, peak_src = tensor_peak()
    print(f"[bench] {w.name}: {ms_step:.3f} ms/step, {value:.1f} TFLOP/s ({timing}), "
          f"e2e {e2e_ms:.3f} ms", file=sys.stderr)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic", "config": {**workload_config(w), "timing": timing},
        "pct_of_peak": 100.0 * value / ws / peak_tf,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": achieved / peak_tf, "peak_source": peak_src,
                     "kernel": f"attn_fwd_bf16_kernel<{w.D}>",
                     "kernel_time": f"{step_ms:.4f} ms per launch ({timing}; the step is this "
                                    f"one kernel)",
                     "traffic": measured_traffic(w.name),
                     "algorithmic_bytes": w.hbm_bytes(),
                     "algorithmic_gbs": w.hbm_bytes() / (step_ms * 1e-3) / 1e9},
        "e2e": {"value": ws * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "call": "attn_fwd_host (pinned host buffers; chunked copies overlapped with the "
                        "kernels)" if host_api else
                        "attn_fwd after pinned host-to-device copies, results copied back"},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "gpu": torch.cuda.get_device_name(dev),
        "system": system_info(dev),
    }
    if warm_ms is not None:
        wt = flops / (warm_ms * 1e-3) / 1e12
        line["warm_l2"] = {"value": wt, "unit": "TFLOP/s", "ms_per_step": warm_ms,
                           "timing": "one CUDA graph of the K steps, inputs in L2"}
    if rank == 0 and not args.no_extra:
        line["workloads"] = extra_workloads(args, dev, stream, local)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, x)
    if rank == 0:
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_backward(args, w):
    """Backward pass alone: device-timed TFLOP/s, 2.5x the forward's FLOPs
    (five matrix products per tile pair instead of two)."""
    import torch
    from exact_io_aware_107_b300 import _binding
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _binding.load()
    x = W.generate(w)
    stream = torch.cuda.current_stream(dev)
    ms, how, clocks, _ = measure_backward(w, x, args.steps, args.warmup, dev, stream, local)
    flops = 2.5 * w.flops()
    peak_tf, peak_src = tensor_peak()
    tf = flops / (ms * 1e-3) / 1e12
    print(f"[bench] backward {w.name}: {ms:.3f} ms/step, {tf:.1f} TFLOP/s", file=sys.stderr)
    line = {
        "metric": "attention bwd TFLOPS (bf16, 2.5x forward FLOPs)", "value": tf,
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "config": {**workload_config(w), "timing": how},
        "roofline": {"bound": "tensor", "achieved": tf, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": tf / peak_tf, "peak_source": peak_src,
                     "kernel": f"attn_bwd_bf16_kernel<{w.D}> (+ prep and dQ kernels)",
                     "traffic": None},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
        "gpu": torch.cuda.get_device_name(dev), "system": system_info(dev),
    }
    print(json.dumps(line))
    return 0


def run_decode(args):
    """KV-cache decode alone: device-timed GB/s against the HBM read roofline."""
    import torch
    from exact_io_aware_107_b300 import _binding
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _binding.load()
    stream = torch.cuda.current_stream(dev)
    shape = tuple(int(t) for t in args.decode_shape.split(","))
    B, H, Nq, Nk, D = shape
    ms, how, clocks, nbytes = measure_decode(shape, args.steps, args.warmup, dev, stream, local)
    nb = decode_bytes(B, H, Nq, Nk, D)
    gbs = nb / (ms * 1e-3) / 1e9
    peak, src = hbm_peak(dev, stream)
    line = {
        "metric": "attention decode GB/s (bf16, KV cache, non-causal)", "value": gbs,
        "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"decode_b{B}_h{H}_nq{Nq}_nk{Nk}_d{D}", "B": B, "H": H, "Nq": Nq,
                   "Nk": Nk, "D": D, "workspace_bytes": nbytes, "timing": how},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                     "frac": gbs / peak, "peak_source": src,
                     "kernel": f"attn_decode_bf16_kernel<{D}>", "traffic": None,
                     "algorithmic_bytes": nb},
        "gpu_launches": args.steps * (2 if nbytes > 0 else 1),
        "clocks": clocks,
        "gpu": torch.cuda.get_device_name(dev), "system": system_info(dev),
    }
    print(json.dumps(line))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=W.HEADLINE,
                    choices=sorted(W.WORKLOADS) + sorted(W.CROSS_WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="leave out the other workloads (key 'workloads' of the line)")
    ap.add_argument("--op", choices=["forward", "backward", "decode"], default="forward",
                    help="backward: dQ, dK, dV (TFLOP/s); decode: the KV-cache decode path "
                         "(GB/s against HBM)")
    ap.add_argument("--decode-shape", default="8,32,1,32768,128", help="B,H,Nq,Nk,D for --op decode")
    ap.add_argument("--shape", default=None,
                    help="B,H,N,D (or B,H,Nq,Nk,D for cross-attention): same dtype and mask "
                         "as --workload at another size (profiling cases)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)   # at least three untimed warm-up steps
    if args.op == "decode":
        return run_decode(args)
    w = {**W.WORKLOADS, **W.CROSS_WORKLOADS}[args.workload]
    if args.shape:
        dims = [int(t) for t in args.shape.split(",")]
        if len(dims) == 4:
            b, h, n, d = dims
            nk = None
            tag = f"n{n}"
        else:
            b, h, n, nk, d = dims
            tag = f"nq{n}_nk{nk}"
        w = W.custom(w.dtype, B=b, H=h, N=n, D=d, causal=w.causal, seed=w.seed, qk_std=w.qk_std,
                     Nk=nk, name=f"{w.dtype}_{'cross_' if nk is not None else ''}"
                                 f"{'causal_' if w.causal else ''}b{b}_h{h}_{tag}_d{d}")
    if args.impl == "reference":
        return run_reference(args, w)
    if args.op == "backward":
        return run_backward(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
