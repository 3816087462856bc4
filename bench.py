"""Throughput of the exact attention forward on B300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline]

A step is one attention forward over the whole workload (default: bf16,
causal, B=2, H=32, N=8192, D=128).  ``value`` is device-timed TFLOP/s with
inputs resident in HBM (CUDA events on the launching stream, K back-to-back
launches; the inputs, 403 MB, exceed the 126 MB L2 so no flush is needed).
``e2e`` is the same metric through the C-ABI call on pinned host buffers
(``attn_fwd_host``): every step copies Q, K, V host->device and O, LSE
device->host inside the timed region, chunk by chunk, overlapped with the
kernels.  Under torchrun each rank runs its own replica of the
workload (weak scaling); the slowest rank's time is used.

``--impl reference`` times the fp64 CPU oracle on the host cores instead,
each step on a bounded sample of the same workload (rank 0 only).
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
    """One BLAS thread per worker thread, when threadpoolctl is available."""
    try:
        from threadpoolctl import threadpool_limits
        return threadpool_limits(limits=1)
    except ImportError:
        import contextlib
        return contextlib.nullcontext()


def _rows_flops(w, rows: np.ndarray) -> float:
    """Attention FLOPs of the given query rows (4 D per allowed key)."""
    nk = w.n_keys
    keys = np.clip(rows + 1 + (nk - w.N), 0, nk) if w.causal else np.full(len(rows), nk)
    return float(4.0 * w.D * keys.sum())


def oracle_rows_sample(w, x, plane_index: int, rows: np.ndarray, threads: int = 1):
    """Run the oracle on the given rows of one plane in this process; returns (flops, seconds)."""
    import oracle
    b, h = divmod(plane_index, w.H)
    q = W.as_f64(x["q"][b, h])
    k = W.as_f64(x["k"][b, h])
    v = W.as_f64(x["v"][b, h])
    with _blas_single_thread():
        t0 = time.perf_counter()
        oracle.attention_rows(q, k, v, w.scale, w.causal, rows)
        dt = time.perf_counter() - t0
    return _rows_flops(w, rows), dt


_ORACLE_PLANE = None


def _oracle_worker_init(q, k, v, scale, causal):
    global _ORACLE_PLANE
    _ORACLE_PLANE = (q, k, v, scale, causal)
    try:
        from threadpoolctl import threadpool_limits
        threadpool_limits(limits=1)
    except ImportError:
        pass


def _oracle_worker_rows(rows):
    import oracle
    q, k, v, scale, causal = _ORACLE_PLANE
    oracle.attention_rows(q, k, v, scale, causal, rows)
    return len(rows)


class OraclePool:
    """The oracle on rows of one plane, row-parallel over spawned processes (one
    BLAS thread each).  Processes, not threads: the per-row NumPy work is too
    small to run in parallel under the interpreter lock.  Spawned, not forked:
    a process forked after CUDA has been initialised can hang."""

    def __init__(self, w, x, plane_index: int, procs: int):
        import multiprocessing as mp
        from concurrent.futures import ProcessPoolExecutor
        b, h = divmod(plane_index, w.H)
        init = (W.as_f64(x["q"][b, h]), W.as_f64(x["k"][b, h]), W.as_f64(x["v"][b, h]),
                w.scale, w.causal)
        self.w, self.x, self.plane, self.procs = w, x, plane_index, procs
        self.ex = ProcessPoolExecutor(max_workers=procs, mp_context=mp.get_context("spawn"),
                                      initializer=_oracle_worker_init, initargs=init)
        # start every worker before anything is timed; a pool that does not come
        # up (a worker that cannot start) falls back to this process alone
        try:
            list(self.ex.map(_oracle_worker_rows, [np.arange(1)] * (2 * procs), timeout=180))
        except Exception:  # noqa: BLE001 - any failure: measure in-process instead
            self.ex.shutdown(wait=False, cancel_futures=True)
            self.ex, self.procs = None, 1

    def run(self, rows: np.ndarray):
        """(flops, seconds) of the oracle on `rows`, dealt round-robin so that
        long and short causal rows spread evenly over the processes."""
        if self.ex is None:
            return oracle_rows_sample(self.w, self.x, self.plane, rows)
        chunks = [rows[i::self.procs] for i in range(self.procs) if len(rows[i::self.procs])]
        t0 = time.perf_counter()
        list(self.ex.map(_oracle_worker_rows, chunks, timeout=600))
        return _rows_flops(self.w, rows), time.perf_counter() - t0

    def close(self):
        if self.ex is not None:
            self.ex.shutdown()


def _sample_block(n: int, done: int, size: int) -> np.ndarray:
    """The next block of the sample: the plane's rows from the last one backwards
    (the full-length causal rows first), starting over once all have been used."""
    r1 = n - (done % n)
    return np.arange(max(0, r1 - size), r1)


def cpu_baseline(w, x, budget_s: float = 12.0):
    """Oracle throughput on a bounded sample: the last rows of plane 0 (full-length causal rows),
    dealt over a process per core; if that turns out slower than one process (a host whose
    cores are shared or throttled), one process on the same budget."""
    procs = host_cores()
    # the same oracle in one process, on the last 256 rows
    one = np.arange(max(0, w.N - 256), w.N)
    f1, dt1 = oracle_rows_sample(w, x, 0, one)
    v1 = f1 / dt1 / 1e12
    pool = OraclePool(w, x, 0, procs)
    try:
        n_rows = 256
        flops_total, t_total, rows_done = 0.0, 0.0, 0
        while t_total < budget_s:
            rows = _sample_block(w.N, rows_done, n_rows)
            f, dt = pool.run(rows)
            flops_total += f
            t_total += dt
            rows_done += len(rows)
            n_rows = min(16384, n_rows * 2)
    finally:
        pool.close()
    procs = pool.procs
    value = flops_total / t_total / 1e12
    how = f"rows dealt over {procs} processes"
    if procs > 1 and value < v1:
        # more processes than the host really runs at once: one process instead
        flops_total, t_total, rows_done, n_rows = 0.0, 0.0, 0, 256
        while t_total < budget_s:
            rows = _sample_block(w.N, rows_done, n_rows)
            f, dt = oracle_rows_sample(w, x, 0, rows)
            flops_total += f
            t_total += dt
            rows_done += len(rows)
            n_rows = min(4096, n_rows * 2)
        how = (f"one process ({procs} processes ran at {value:.2e} TFLOP/s, below one "
               f"process: the host's cores are shared or throttled)")
        value, procs = flops_total / t_total / 1e12, 1
    return {"value": value, "unit": "TFLOP/s", "cores": procs,
            "kind": "oracle", "value_1core": v1,
            "sample": f"fp64 oracle on {rows_done} query rows of plane (b=0,h=0) of "
                      f"{w.name} (from the last row backwards, starting over after row 0), "
                      f"{how} ({t_total:.1f} s); "
                      f"value_1core: the last {len(one)} rows in one process ({dt1:.2f} s)"}


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    x = W.generate(w)
    threads = host_cores()
    rows = np.arange(max(0, w.N - 512), w.N)   # one step: the last 512 rows of plane 0
    pool = OraclePool(w, x, 0, threads)
    try:
        # a process per core, unless that is slower than one process on this host
        _, t_one = oracle_rows_sample(w, x, 0, rows)
        _, t_pool = pool.run(rows)
        step = pool.run if t_pool < t_one else (lambda r: oracle_rows_sample(w, x, 0, r))
        threads = pool.procs if t_pool < t_one else 1
        for _ in range(args.warmup):
            step(rows)
        flops = secs = 0.0
        for _ in range(args.steps):
            f, dt = step(rows)
            flops += f
            secs += dt
    finally:
        pool.close()
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"each step: fp64 oracle on query rows {rows[0]}..{rows[-1]} "
                                   f"of plane (b=0,h=0) of {w.name}, dealt over {threads} "
                                   f"process(es)"},
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
    q, k, v = (t.to(dev) for t in (x["q"], x["k"], x["v"]))
    cu = None if x["cu_seqlens"] is None else torch.as_tensor(x["cu_seqlens"]).to(dev)
    cuk = None if x["cu_seqlens_k"] is None else torch.as_tensor(x["cu_seqlens_k"]).to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = None
    if 3 * w.hbm_bytes() / 4 <= 126e6:
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        if flush is not None:
            flush.zero_()
        attention_forward(q, k, v, causal=w.causal, scale=w.scale, cu_seqlens=cu, out=o, lse=lse,
                          stream=stream, cu_seqlens_k=cuk)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if device_error() != 0:
        raise RuntimeError("device error during warm-up")

    # --- device-timed region (inputs resident) ---
    # Without a flush the K steps are also captured into one CUDA graph and the
    # graph's replay is what `value` times: the same kernels back to back, with
    # no host launch gaps in between.
    graph = None
    if flush is None:
        try:
            graph = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream(dev)
            cap.wait_stream(stream)
            with torch.cuda.graph(graph, stream=cap):
                for _ in range(args.steps):
                    attention_forward(q, k, v, causal=w.causal, scale=w.scale, cu_seqlens=cu,
                                      out=o, lse=lse, cu_seqlens_k=cuk)
            stream.wait_stream(cap)
            graph.replay()
            torch.cuda.synchronize()
        except Exception as e:  # noqa: BLE001 - fall back to the eager region
            print(f"[bench] graph capture failed ({e}); timing the eager launches", file=sys.stderr)
            graph = None
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(args.steps):
            if flush is not None:
                flush.zero_()
            starts[i].record(stream)
            attention_forward(q, k, v, causal=w.causal, scale=w.scale, cu_seqlens=cu, out=o,
                              lse=lse, stream=stream, cu_seqlens_k=cuk)
            ends[i].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        if graph is not None:
            g0 = torch.cuda.Event(enable_timing=True)
            g1 = torch.cuda.Event(enable_timing=True)
            barrier(ws)
            with torch.cuda.stream(stream):
                g0.record(stream)
                graph.replay()
                g1.record(stream)
            torch.cuda.synchronize()
    barrier(ws)
    if device_error() != 0:
        raise RuntimeError("device error in the timed region")
    total_ms = t_start.elapsed_time(t_end)
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    kernel_ms = sum(launch_ms) / len(launch_ms)
    # with an L2 flush between launches the step is the attention call alone
    # (the events bracket it); otherwise the K steps of the graph replay
    warm = None
    if flush is not None:
        step_ms, timing = kernel_ms, "per-launch CUDA events, L2 flushed between launches"
        # the same workload warm in L2: the K steps back to back in one CUDA graph
        warm_ms = graph_step_ms(
            lambda st: attention_forward(q, k, v, causal=w.causal, scale=w.scale, cu_seqlens=cu,
                                         out=o, lse=lse, stream=st, cu_seqlens_k=cuk),
            args.steps, stream, dev)
        if warm_ms is not None:
            warm = {"value": w.flops() / (warm_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "ms_per_step": warm_ms, "timing": "one CUDA graph of the K steps, inputs in L2"}
    elif graph is not None:
        step_ms, timing = g0.elapsed_time(g1) / args.steps, "one CUDA graph of the K steps"
    else:
        step_ms, timing = total_ms / args.steps, "K eager launches back to back"
    ms_step = max_over_ranks(step_ms, ws)
    flops = w.flops()
    value = ws * flops / (ms_step * 1e-3) / 1e12

    # --- end-to-end region: pinned host buffers, copies inside the timed region ---
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

    peak_tf, _, peak_kind = load_peaks()
    achieved = flops / (kernel_ms * 1e-3) / 1e12
    print(f"[bench] {w.name}: {ms_step:.3f} ms/step, {value:.1f} TFLOP/s, kernel {kernel_ms:.3f} ms"
          f" ({achieved:.1f} TFLOP/s), e2e {e2e_ms:.3f} ms", file=sys.stderr)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic", "config": {**workload_config(w), "timing": timing},
        "pct_of_peak": 100.0 * value / ws / peak_tf,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": achieved / peak_tf,
                     "peak_source": f"{peak_kind} cuBLAS bf16 burst (MEASURED_PEAKS.json)"
                     if peak_kind == "measured" else "fallback 1.8 PFLOP/s",
                     "kernel": f"attn_fwd_bf16_kernel<{w.D}>",
                     "traffic": measured_traffic(w.name),
                     "algorithmic_bytes": w.hbm_bytes(),
                     "algorithmic_gbs": w.hbm_bytes() / (kernel_ms * 1e-3) / 1e9},
        "e2e": {"value": ws * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "call": "attn_fwd_host (pinned host buffers; chunked copies overlapped with the "
                        "kernels)" if host_api else
                        "attn_fwd after pinned host-to-device copies, results copied back"},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
        "gpu": torch.cuda.get_device_name(dev),
        "system": system_info(dev),
    }
    if warm is not None:
        line["warm_l2"] = warm
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, x)
    if rank == 0:
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def graph_step_ms(step, steps, stream, dev):
    """Milliseconds per step of `steps` calls of step() captured into one CUDA
    graph and replayed (the same kernels back to back, without host launch
    gaps); None when the capture is refused."""
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
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps
    except Exception as e:  # noqa: BLE001 - the caller falls back to eager timing
        print(f"[bench] graph capture failed ({e})", file=sys.stderr)
        return None


def run_backward(args, w):
    """Backward pass (a NEXT row): device-timed TFLOP/s, 2.5x the forward's FLOPs
    (five matrix products per tile pair instead of two)."""
    import torch
    from exact_io_aware_107_b300 import (_binding, attention_backward, attention_forward,
                                         device_error)

    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _binding.load()
    x = W.generate(w)
    q, k, v = (t.to(dev) for t in (x["q"], x["k"], x["v"]))
    rng = np.random.default_rng(1)
    do = torch.from_numpy(rng.standard_normal(tuple(q.shape), dtype=np.float32)).to(q.dtype).to(dev)
    cu = None if x["cu_seqlens"] is None else torch.as_tensor(x["cu_seqlens"]).to(dev)
    cuk = None if x["cu_seqlens_k"] is None else torch.as_tensor(x["cu_seqlens_k"]).to(dev)
    stream = torch.cuda.current_stream(dev)
    o, lse = attention_forward(q, k, v, causal=w.causal, scale=w.scale, cu_seqlens=cu,
                               cu_seqlens_k=cuk, stream=stream)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    rc, nbytes = _binding.attn_bwd_workspace_bytes(w.B, w.H, w.N, w.D, cu is not None)
    assert rc == 0
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)

    def step(st=stream):
        attention_backward(q, k, v, o, lse, do, causal=w.causal, scale=w.scale, cu_seqlens=cu,
                           cu_seqlens_k=cuk, dq=dq, dk=dk, dv=dv, workspace=ws, stream=st)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if device_error() != 0:
        raise RuntimeError("device error during warm-up")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        g_ms = graph_step_ms(step, args.steps, stream, dev)
    if device_error() != 0:
        raise RuntimeError("device error in the timed region")
    eager_ms = sum(s_.elapsed_time(e) for s_, e in zip(starts, ends)) / args.steps
    ms = g_ms if g_ms is not None else eager_ms
    flops = 2.5 * w.flops()
    peak_tf, _, peak_kind = load_peaks()
    tf = flops / (ms * 1e-3) / 1e12
    print(f"[bench] backward {w.name}: {ms:.3f} ms/step, {tf:.1f} TFLOP/s", file=sys.stderr)
    line = {
        "metric": "attention bwd TFLOPS (bf16, 2.5x forward FLOPs)", "value": tf,
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {**workload_config(w),
                   "l2": "inputs larger than L2 (no flush)" if 5 * w.hbm_bytes() / 4 > 126e6
                   else "inputs smaller than L2 (not flushed)",
                   "timing": "one CUDA graph of the K steps" if g_ms is not None
                   else "per-step CUDA events"},
        "roofline": {"bound": "tensor", "achieved": tf, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": tf / peak_tf, "peak_source": f"{peak_kind} cuBLAS bf16 burst",
                     "kernel": f"attn_bwd_bf16_kernel<{w.D}> (+ prep and dQ kernels)",
                     "traffic": None},
        "gpu_launches": 3 * args.steps,
        "clocks": clk.summary(),
        "gpu": torch.cuda.get_device_name(dev), "system": system_info(dev),
    }
    print(json.dumps(line))
    return 0


def run_decode(args):
    """KV-cache decode (a NEXT row): device-timed GB/s against the HBM roofline."""
    import torch
    from exact_io_aware_107_b300 import _binding, attention_decode, device_error

    ws_, rank, local = dist_env()
    torch.cuda.set_device(local)
    B, H, Nq, Nk, D = (int(t) for t in args.decode_shape.split(","))
    rng = np.random.default_rng(0)
    def draw(*shape):
        return torch.from_numpy(rng.standard_normal(shape, dtype=np.float32)).to(torch.bfloat16)
    q, k, v = draw(B, H, Nq, D), draw(B, H, Nk, D), draw(B, H, Nk, D)
    dev = torch.device("cuda", local)
    dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
    rc, nbytes = _binding.attn_decode_workspace_bytes(B, H, Nq, Nk, D)
    assert rc == 0
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    o = torch.empty_like(dq)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        attention_decode(dq, dk, dv, workspace=ws, out=o, lse=lse, stream=stream)
    torch.cuda.synchronize()
    assert device_error() == 0
    with ClockSampler(local) as clk:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            attention_decode(dq, dk, dv, workspace=ws, out=o, lse=lse, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        g_ms = graph_step_ms(lambda st: attention_decode(dq, dk, dv, workspace=ws, out=o, lse=lse,
                                                         stream=st),
                             args.steps, stream, dev)
    assert device_error() == 0
    ms = g_ms if g_ms is not None else e0.elapsed_time(e1) / args.steps
    nbytes_alg = 2 * B * H * Nk * D * 2 + 2 * B * H * Nq * D * 2 + B * H * Nq * 4
    _, hbm_peak, kind = load_peaks()
    gbs = nbytes_alg / (ms * 1e-3) / 1e9
    line = {
        "metric": "attention decode GB/s (bf16, KV cache, non-causal)", "value": gbs,
        "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"decode_b{B}_h{H}_nq{Nq}_nk{Nk}_d{D}", "B": B, "H": H, "Nq": Nq,
                   "Nk": Nk, "D": D, "workspace_bytes": nbytes,
                   "timing": "one CUDA graph of the K steps" if g_ms is not None
                   else "K launches back to back",
                   "l2": "K/V larger than L2 (no flush)" if 2 * B * H * Nk * D * 2 > 126e6
                   else "K/V fit in L2"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                     "frac": gbs / hbm_peak, "peak_source": f"{kind} copy bandwidth",
                     "kernel": f"attn_decode_bf16_kernel<{D}>", "traffic": None,
                     "algorithmic_bytes": nbytes_alg},
        "gpu_launches": args.steps * (2 if nbytes > 0 else 1),
        "clocks": clk.summary(),
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
