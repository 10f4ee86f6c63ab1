"""Benchmark of the row-reduction kernels: effective HBM TB/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one call of the operator over one batch (the full M x N matrix of
the workload) with its inputs already resident in HBM.  The metric is the
effective memory throughput: the minimal bytes the operator must move (read
every input once, write every output once) divided by the device time.

Timing: W warm-up steps, then K steps between CUDA events on the launching
stream, with a barrier and synchronize on both sides; the max over ranks is
taken.  The K steps are issued twice, in two timed regions: once as a CUDA
graph of the K calls, replayed once (the headline: no host launch overhead
between steps, as a launch-bound loop is issued in production), and once call
by call from Python (reported beside it).  Before each timed region a spin
kernel holds the stream for ~0.5 ms, so that the calls are enqueued before
the GPU reaches the start event; in the graph the two events are nodes
recorded right before the first call and after the last, so the events
measure device time only.  Inputs are larger than 4x the L2
size, or input/output sets rotate over more than that, so no step finds its
data in L2.  SM clocks and throttle reasons are sampled with nvidia-smi for
the whole run; each entry reports the samples taken from its warm-up to the
end of a 0.3 s hold of the same steps, untimed, right after its timed regions
(a K-step region of tens of microseconds is shorter than the sampling period).

With one GPU the line also carries, at the same K and W:
  per_workload  the other named workloads (softmax 1024 x 4096 fp32,
                cross-entropy 8192 x 131072 bf16, softmax 16384 x 131072 fp32)
                and the backward / LayerNorm workloads, each with its roofline;
  sweep         the M x N sweep (3 operators x fp32/bf16 x M x N), per
                operator and dtype the min and median fraction of peak over
                N >= 4096 and the worst point, and every point.

Multi-GPU (torchrun, one rank per GPU): rows are independent, so each rank
processes its own batch of the same shape (weak scaling, no collective on the
data path; one max-reduction of the elapsed time after the timed region).

--impl reference times the fp64 CPU oracle on the host cores instead (rank 0
only), each step a bounded sample of rows of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from memory_bound_row_rmsnorm_gb300 import synthetic as syn  # noqa: E402

L2_BYTES = 129 * 10 ** 6
FALLBACK_HBM_GBS = 6800.0
# GB300 HBM3e data sheet bandwidth, reported beside the measured copy peak.
NOMINAL_HBM_GBS = 7900.0
METRIC = "effective HBM TB/s and % of GB300 peak per kernel over the M×N sweep"
ESIZE = {"f32": 4, "bf16": 2}
DEFAULT_WORKLOAD = "rmsnorm_bf16_16384x4096"
EPS = 1e-6
OP_CODES = {"softmax": 0, "rmsnorm": 1, "xent": 2, "softmax_bwd": 3, "rmsnorm_bwd": 4, "xent_bwd": 5,
            "layernorm": 6}


def min_bytes(op: str, dtype: str, M: int, N: int) -> int:
    """Algorithmic bytes of one call: every input read once, every output written once."""
    s = ESIZE[dtype]
    if op == "softmax":
        return 2 * M * N * s
    if op == "rmsnorm":
        return 2 * M * N * s + N * s + 4 * M
    if op == "xent":
        return M * N * s + 8 * M + 8 * M  # logits + targets in; loss + lse out
    if op == "softmax_bwd":
        return 3 * M * N * s  # y, dy in; dx out
    if op == "rmsnorm_bwd":
        return 3 * M * N * s + N * s + 4 * M + 4 * N  # x, dy, w, rstd in; dx, dw out
    if op == "xent_bwd":
        return 2 * M * N * s + 16 * M  # logits, targets, lse, dloss in; dlogits out
    if op == "layernorm":
        return 2 * M * N * s + 2 * N * s + 8 * M  # x, w, b in; y, mean, rstd out
    raise ValueError(op)


# The device code of the kernels (the launch plan is compared separately).
KERNEL_SOURCES = ("qk_device.cuh", "qk_kernels.cuh", "qk_kernel_table.cuh", "qk_internal.h",
                  "qk_bwd_kernels.cuh", "qk_bwd_table.cuh")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    d = os.path.join(ROOT, "memory_bound_row_rmsnorm_gb300", "csrc")
    for f in KERNEL_SOURCES:
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs, copy burst)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (no MEASURED_PEAKS.json)"


def recorded_traffic(workload: str, plan: dict):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources with the same launch plan; otherwise None."""
    p = os.path.join(ROOT, "profiles", f"{workload}.traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("kernel_source_hash") != kernel_source_hash():
        return None
    keys = ("threads", "row_threads", "vec_per_thread", "cluster", "slots", "chunks")
    if any(rec.get("plan", {}).get(k) != plan.get(k) for k in keys):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while running.
    Each sample carries nvidia-smi's own timestamp, so a summary can be taken
    over the samples of one time window (host wall clock, time.time())."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        cmd = ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
               "--format=csv,noheader,nounits", "-lms", "100"]
        # line-buffered output through a pipe when stdbuf is there, so that
        # every sample reaches the reader as it is taken
        for prefix in (["stdbuf", "-oL"], []):
            try:
                self.proc = subprocess.Popen(prefix + cmd, stdout=subprocess.PIPE,
                                             stderr=subprocess.DEVNULL, text=True)
                break
            except Exception:
                self.proc = None
        if self.proc is not None:
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self._t.join(timeout=2)

    @staticmethod
    def _stamp(field: str):
        """Seconds since the epoch of an nvidia-smi timestamp (local time), or None."""
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(field.strip(), fmt).timestamp()
            except ValueError:
                continue
        return None

    def summary(self, t0: float | None = None, t1: float | None = None):
        """Median SM clock, max clock, throttle reasons and sample count, over
        every sample or over those stamped inside [t0, t1]."""
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            ts = self._stamp(parts[0]) if parts else None
            if ts is not None:
                parts = parts[1:]
            if len(parts) < 9:
                continue
            if t0 is not None and (ts is None or ts < t0 or ts > t1):
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_seed(rank: int, i: int) -> int:
    """Seed of input set i on `rank`: every rank draws its own rows."""
    return 1000 + 17 * rank + i


def max_over_ranks(value: float, dist, device) -> float:
    """The largest of `value` over all ranks (the job ends with its slowest rank)."""
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tbs(bytes_per_rank_step: int, world: int, steps: int, ms: float) -> float:
    """Whole-job throughput: all ranks' algorithmic bytes over the slowest rank's time."""
    return bytes_per_rank_step * world * steps / (ms / 1e3) / 1e12


def make_set(op, dtype, M, N, sigma, seed, dev):
    inp = syn.make_inputs(op, dtype, M, N, seed, dev, sigma)
    out = {}
    if op.endswith("_bwd"):
        ref = inp["y"] if op == "softmax_bwd" else inp["x"]
        out["dx"] = torch.empty_like(ref)
        if op == "rmsnorm_bwd":
            from memory_bound_row_rmsnorm_gb300 import binding as qb
            nbytes = qb.qk_rmsnorm_bwd_workspace_size(M, N, qb.QK_F32 if dtype == "f32" else qb.QK_BF16)
            out["dw"] = torch.empty(N, dtype=torch.float32, device=dev)
            out["workspace"] = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
        return inp, out
    if op in ("softmax", "rmsnorm", "layernorm"):
        out["y"] = torch.empty_like(inp["x"])
    if op in ("rmsnorm", "layernorm"):
        out["rstd"] = torch.empty(M, dtype=torch.float32, device=dev)
    if op == "layernorm":
        out["mean"] = torch.empty(M, dtype=torch.float32, device=dev)
    if op == "xent":
        out["loss"] = torch.empty(M, dtype=torch.float32, device=dev)
        out["lse"] = torch.empty(M, dtype=torch.float32, device=dev)
    return inp, out


def launch(qb, op, dtype, inp, out, M, N, stream):
    code = qb.QK_F32 if dtype == "f32" else qb.QK_BF16
    if op == "softmax_bwd":
        qb.qk_softmax_bwd(inp["y"], inp["dy"], out["dx"], M, N, code, stream)
    elif op == "rmsnorm_bwd":
        ws = out["workspace"]
        qb.qk_rmsnorm_bwd(inp["x"], inp["w"], inp["rstd"], inp["dy"], out["dx"], out["dw"], ws,
                          ws.numel(), M, N, code, stream)
    elif op == "xent_bwd":
        qb.qk_xent_bwd(inp["x"], inp["targets"], inp["lse"], inp["dloss"], out["dx"], M, N, code, stream)
    elif op == "softmax":
        qb.qk_softmax_fwd(inp["x"], out["y"], M, N, code, stream)
    elif op == "rmsnorm":
        qb.qk_rmsnorm_fwd(inp["x"], inp["w"], out["y"], out["rstd"], M, N, EPS, code, stream)
    elif op == "layernorm":
        qb.qk_layernorm_fwd(inp["x"], inp["w"], inp["b"], out["y"], out["mean"], out["rstd"], M, N,
                            EPS, code, stream)
    else:
        qb.qk_xent_fwd(inp["x"], inp["targets"], out["loss"], out["lse"], M, N, code, stream)


HEAD_START_CYCLES = 1_000_000  # about 0.5 ms of SM cycles at 2 GHz


def head_start(stream) -> None:
    """Keeps `stream` busy for about half a millisecond (torch's spin kernel,
    before the start event) so that the timed calls are already enqueued when
    the GPU reaches the start event: the two events then bracket device time
    only, not the host's submission of the first calls or of the graph."""
    with torch.cuda.stream(stream):
        torch.cuda._sleep(HEAD_START_CYCLES)


def timed_launches(qb, op, dtype, sets, M, N, K, stream, graph: bool, dev):
    """Enqueues K steps (rotating over `sets`) between two CUDA events on
    `stream` and returns (start, stop).  With graph=True the K calls are first
    captured into one CUDA graph (the library's launches, recorded once) and
    the graph is replayed, which removes host launch overhead between steps;
    the two events are then nodes of the graph itself, recorded right before
    the first call and right after the last, so that the graph's own launch
    is not counted.  Either way one untimed pass over every set, in the
    order the timed steps take them, comes first, so that each timed step's
    set was last touched len(sets) steps earlier (none is still in L2 from an
    earlier pass), and a head start (head_start) precedes the timed region."""
    nsets = len(sets)

    def rotate():
        for i in range(nsets):
            inp, out = sets[i]
            launch(qb, op, dtype, inp, out, M, N, stream)

    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if not graph:
        rotate()
        head_start(stream)
        start.record(stream)
        for i in range(K):
            inp, out = sets[i % nsets]
            launch(qb, op, dtype, inp, out, M, N, stream)
        stop.record(stream)
        return start, stop
    start = torch.cuda.Event(enable_timing=True, external=True)
    stop = torch.cuda.Event(enable_timing=True, external=True)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream(dev)
        start.record(cs)
        for i in range(K):
            inp, out = sets[i % nsets]
            launch(qb, op, dtype, inp, out, M, N, cs)
        stop.record(cs)
    g.replay()  # first replay uploads the graph
    torch.cuda.synchronize(dev)
    rotate()
    head_start(stream)
    g.replay()
    timed_launches.keep = g  # the graph must outlive the replay
    return start, stop


def e2e_pipelined(qb, op, dtype, dev_sets, M, N, steps, dev):
    """End-to-end steps through the public API with HOST buffers: every step
    copies its inputs from pinned host memory to the device, calls the
    operator, and copies its outputs back to pinned host memory.  Steps are
    pipelined over three streams (copy-in, compute, copy-out) and two device
    buffer sets, so step i's copy-out overlaps step i+1's copy-in and kernel;
    events keep each device buffer from being overwritten while in use.
    Returns (elapsed ms, steps, h2d bytes per step, d2h bytes per step)."""
    inp0, out0 = dev_sets[0]
    h_in = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True).copy_(v) for k, v in inp0.items()}
    h_out = [{k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in o.items()}
             for _, o in dev_sets]
    h2d = sum(v.numel() * v.element_size() for v in h_in.values())
    d2h = sum(v.numel() * v.element_size() for v in h_out[0].values())
    s_in, s_run, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    nb = len(dev_sets)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    loaded = [ev() for _ in range(nb)]    # inputs of set b are on the device
    computed = [ev() for _ in range(nb)]  # kernel on set b finished (inputs free, outputs ready)
    drained = [ev() for _ in range(nb)]   # outputs of set b copied to the host (outputs free)

    def run(n):
        for i in range(n):
            b = i % nb
            inp, out = dev_sets[b]
            if i >= nb:
                s_in.wait_event(computed[b])
            with torch.cuda.stream(s_in):
                for k in inp:
                    inp[k].copy_(h_in[k], non_blocking=True)
                loaded[b].record(s_in)
            s_run.wait_event(loaded[b])
            if i >= nb:
                s_run.wait_event(drained[b])
            launch(qb, op, dtype, inp, out, M, N, s_run)
            computed[b].record(s_run)
            s_out.wait_event(computed[b])
            with torch.cuda.stream(s_out):
                for k in out:
                    h_out[b][k].copy_(out[k], non_blocking=True)
                drained[b].record(s_out)

    cur = torch.cuda.current_stream(dev)
    run(2)
    torch.cuda.synchronize(dev)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(cur)
    for s_ in (s_in, s_run, s_out):
        s_.wait_stream(cur)
    run(steps)
    for s_ in (s_in, s_run, s_out):
        cur.wait_stream(s_)
    stop.record(cur)
    torch.cuda.synchronize(dev)
    return start.elapsed_time(stop), steps, h2d, d2h


def oracle_inputs(op, dtype, rows, N, sigma, seed):
    """Seeded rows of the workload, widened to float64 for the oracle."""
    inp = syn.make_inputs(op, dtype, rows, N, seed, "cpu", sigma)
    return {k: (v.numpy() if v.dtype == torch.int64 else v.to(torch.float64).numpy()) for k, v in inp.items()}


def oracle_call(oracle, lib, op, d, sl):
    """The oracle (as it stands) on rows `sl` of the inputs `d`."""
    if op == "softmax":
        oracle.softmax_fwd(d["x"][sl], lib)
    elif op == "rmsnorm":
        oracle.rmsnorm_fwd(d["x"][sl], d["w"], EPS, lib)
    elif op == "xent":
        oracle.xent_fwd(d["x"][sl], d["targets"][sl], lib)
    elif op == "softmax_bwd":
        oracle.softmax_bwd(d["y"][sl], d["dy"][sl], lib)
    elif op == "rmsnorm_bwd":
        oracle.rmsnorm_bwd(d["x"][sl], d["w"], d["rstd"][sl], d["dy"][sl], lib)
    elif op == "layernorm":
        oracle.layernorm_fwd(d["x"][sl], d["w"], d["b"], EPS, lib)
    else:
        oracle.xent_bwd(d["x"][sl], d["targets"][sl], d["lse"][sl], d["dloss"][sl], lib)


def cpu_oracle_rate(op, dtype, M, N, sigma, budget_s: float, seed: int = 4242):
    """The fp64 oracle, as it stands, over seeded rows of the workload on all
    host cores (one thread per core, each running the oracle on its own rows).
    Returns (TB/s, cores, sample description, seconds)."""
    import concurrent.futures as cf

    import oracle

    cores = os.cpu_count() or 1
    lib = oracle.library()
    # enough rows per thread that each call spends its time in the C oracle,
    # not in the Python around it (ctypes releases the GIL only inside the
    # call); at most 2^27 elements held in float64
    rows = min(M, max(cores * 128, 256), max(cores, (1 << 27) // N))
    d = oracle_inputs(op, dtype, rows, N, sigma, seed)
    parts = [p for p in np.array_split(np.arange(rows), cores) if p.size]

    def work(idx):
        oracle_call(oracle, lib, op, d, slice(int(idx[0]), int(idx[-1]) + 1))

    reps = 0
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        list(ex.map(work, parts))  # warm
        t0 = time.perf_counter()
        while True:
            list(ex.map(work, parts))
            reps += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                break
    nbytes = min_bytes(op, dtype, rows, N) * reps
    sample = (f"{reps} passes over {rows} seeded rows x {N} of the workload "
              f"({rows * reps} rows, {el:.1f} s), {cores} threads")
    return nbytes / el / 1e12, cores, sample, el


def cpu_single_core_rate(op, dtype, N, sigma, budget_s: float, seed: int = 4243):
    """The same oracle on one thread of the host (the per-core rate)."""
    import oracle

    lib = oracle.library()
    rows = 64
    d = oracle_inputs(op, dtype, rows, N, sigma, seed)
    oracle_call(oracle, lib, op, d, slice(0, rows))  # warm
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle_call(oracle, lib, op, d, slice(0, rows))
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return min_bytes(op, dtype, rows, N) * reps / el / 1e12


def cpu_model() -> str:
    """The host CPU's name as the kernel reports it (x86 and Arm layouts)."""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
    except OSError:
        return platform.machine()
    for key in ("model name", "Model Name", "Hardware"):
        for line in info.splitlines():
            if line.split(":")[0].strip() == key:
                return line.split(":", 1)[1].strip()
    parts = sorted({line.split(":", 1)[1].strip() for line in info.splitlines()
                    if line.split(":")[0].strip() == "CPU part"})
    return f"{platform.machine()} (CPU part {', '.join(parts)})" if parts else platform.machine()


def run_reference(args, op, dtype, M, N, sigma):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle  # noqa: F401  (builds the C oracle on first use)

    K, W = args.steps, args.warmup
    # calibrate rows per step so the whole run stays within ~2 minutes
    rate, cores, _, _ = cpu_oracle_rate(op, dtype, M, N, sigma, budget_s=min(1.0, args.ref_seconds / 4))
    per_row = min_bytes(op, dtype, 1, N)
    budget = args.ref_seconds / max(1, K + W)
    rows = int(max(1, min(M, rate * 1e12 * budget / per_row)))
    import concurrent.futures as cf

    lib = oracle.library()
    d = oracle_inputs(op, dtype, rows, N, sigma, 4343)
    parts = [p for p in np.array_split(np.arange(rows), cores) if p.size]

    def work(idx):
        oracle_call(oracle, lib, op, d, slice(int(idx[0]), int(idx[-1]) + 1))

    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        for _ in range(W):
            list(ex.map(work, parts))
        t0 = time.perf_counter()
        for _ in range(K):
            list(ex.map(work, parts))
        el = time.perf_counter() - t0
    value = min_bytes(op, dtype, rows, N) * K / el / 1e12
    sample = f"each step: {rows} seeded rows x {N} of the workload on {cores} threads"
    line = {
        "metric": METRIC, "value": value, "unit": "TB/s", "n_gpus": ws, "steps": K, "warmup": W,
        "ms_per_step": el / K * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "op": op, "M": M, "N": N, "input_dtype": dtype,
                   "rows_per_step": rows},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "TB/s", "cores": cores, "kind": "oracle",
                         "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


HOLD_S = 0.3  # untimed hold after each entry's timed regions, so that its clock record has samples
# A K-step graph region shorter than this is timed once more, with enough steps
# to last about LONG_TARGET_MS: the same kernel's rate once the region's one-off
# costs (its first launch, which no earlier kernel overlaps; the event pair) are
# spread over many calls.  Reported beside the K-step number, never instead of it.
LONG_REGION_MS = 2.0
LONG_TARGET_MS = 4.0
LONG_MAX_STEPS = 2000
ALL_WORKLOADS = {**syn.WORKLOADS, **syn.BWD_WORKLOADS, **syn.NEXT_WORKLOADS}


def n_sets(set_bytes: int) -> int:
    """Input/output sets to rotate over so that no step finds its data in L2:
    one when a set alone is over 4x L2, else enough to pass 4x L2 together."""
    return 1 if set_bytes >= 4 * L2_BYTES else max(2, math.ceil(4 * L2_BYTES / set_bytes))


def kernels_per_step(op: str) -> int:
    """Kernels of the library one call launches (RMSNorm backward: the ring
    kernel, then the fixed-order sum of the dw partials)."""
    return 2 if op == "rmsnorm_bwd" else 1


def hold(qb, op, dtype, sets, M, N, stream, dev, seconds: float, per_launch_ms: float):
    """Keeps issuing the same steps, untimed, for about `seconds`, in batches
    of ~20 ms of GPU work so the queue stays short and the hold ends on time."""
    batch = int(max(8, min(4096, 20.0 / max(per_launch_ms, 1e-3))))
    t_end, i = time.time() + seconds, 0
    while time.time() < t_end:
        for _ in range(batch):
            inp, out = sets[i % len(sets)]
            launch(qb, op, dtype, inp, out, M, N, stream)
            i += 1
        torch.cuda.synchronize(dev)


def time_entry(qb, op, dtype, M, N, sigma, K, W, dev, stream, seed=77, hold_s=HOLD_S,
               modes=("graph", "stream"), long_region=False):
    """W warm-up steps, then K steps timed once per launch mode, then an untimed
    hold.  Returns ({mode: ms per step}, (start of the warm-up, end of the
    hold), {"t0", "t1"} of the timed regions), the times from time.time().
    With long_region, a graph region of K steps that lasts under
    LONG_REGION_MS is timed once more with enough steps to last about
    LONG_TARGET_MS: ms["graph_long"] = (steps, ms per step)."""
    sb = min_bytes(op, dtype, M, N)
    sets = [make_set(op, dtype, M, N, sigma, seed + i, dev) for i in range(n_sets(sb))]
    torch.cuda.synchronize(dev)
    t_start = time.time()
    for i in range(W):
        launch(qb, op, dtype, *sets[i % len(sets)], M, N, stream)
    torch.cuda.synchronize(dev)
    ms = {}
    t0 = time.time()
    for mode in modes:
        e0, e1 = timed_launches(qb, op, dtype, sets, M, N, K, stream, mode == "graph", dev)
        torch.cuda.synchronize(dev)
        ms[mode] = e0.elapsed_time(e1) / K
    per_step = min(ms.values())
    if long_region and "graph" in ms and K * ms["graph"] < LONG_REGION_MS:
        KL = min(LONG_MAX_STEPS, max(K, math.ceil(LONG_TARGET_MS / ms["graph"])))
        e0, e1 = timed_launches(qb, op, dtype, sets, M, N, KL, stream, True, dev)
        torch.cuda.synchronize(dev)
        ms["graph_long"] = (KL, e0.elapsed_time(e1) / KL)
    t1 = time.time()
    if hold_s > 0:
        hold(qb, op, dtype, sets, M, N, stream, dev, hold_s, per_step)
    t_end = time.time()
    st = qb.qk_get_device_status(stream)
    if st != qb.QK_OK:
        raise RuntimeError(f"device status after {op} {dtype} {M}x{N}: {qb.qk_status_string(st)}")
    del sets
    torch.cuda.empty_cache()
    return ms, (t_start, t_end), {"t0": t0, "t1": t1}


def tbs_of(op, dtype, M, N, ms: float) -> float:
    return min_bytes(op, dtype, M, N) / (ms * 1e-3) / 1e12


def roofline(op, dtype, M, N, ms, peak, peak_src, traffic=None) -> dict:
    """The HBM roofline of one call: algorithmic bytes over its device time."""
    b = min_bytes(op, dtype, M, N)
    gbs = b / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
            "traffic": traffic, "peak_source": peak_src, "bytes_per_launch": b,
            "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": gbs / NOMINAL_HBM_GBS}


def workload_entry(qb, name, K, W, dev, stream, peak, peak_src) -> dict:
    """One named workload at K steps: graph and call-by-call rates, roofline and
    the launch plan; "clocks" holds the entry's time window until the sampler
    has stopped (finish_clocks)."""
    op, dtype, M, N, sigma = ALL_WORKLOADS[name]
    ms, window, _ = time_entry(qb, op, dtype, M, N, sigma, K, W, dev, stream, long_region=True)
    code = qb.QK_F32 if dtype == "f32" else qb.QK_BF16
    plan = qb.qk_get_plan(OP_CODES[op], code, M, N)
    g, s = ms["graph"], ms["stream"]
    entry = {
        "workload": name, "op": op, "dtype": dtype, "M": M, "N": N, "steps": K, "warmup": W,
        "ms_per_step": g, "value": tbs_of(op, dtype, M, N, g), "unit": "TB/s", "launch": "cuda_graph",
        "stream": {"ms_per_step": s, "value": tbs_of(op, dtype, M, N, s),
                   "frac": tbs_of(op, dtype, M, N, s) * 1e3 / peak},
        "roofline": roofline(op, dtype, M, N, g, peak, peak_src, recorded_traffic(name, plan)),
        "gpu_launches": K * kernels_per_step(op), "clocks": window, "plan": plan,
    }
    if "graph_long" in ms:
        entry["long_region"] = long_region_entry(op, dtype, M, N, *ms["graph_long"], peak)
    return entry


def long_region_entry(op, dtype, M, N, steps, ms_step, peak) -> dict:
    return {"steps": steps, "ms_per_step": ms_step, "value": tbs_of(op, dtype, M, N, ms_step),
            "frac": tbs_of(op, dtype, M, N, ms_step) * 1e3 / peak,
            "how": "the same calls as one graph of this many steps (a region of about "
                   f"{LONG_TARGET_MS:g} ms), timed after the K-step regions"}


def region_floor_ms(dev, stream, reps: int = 5) -> float:
    """Device time between the two events of an empty timed region (a graph
    holding only the event pair, replayed after a head start): the part of
    every graph-timed number that no kernel can remove.  Median of reps."""
    ts = []
    for _ in range(reps):
        start = torch.cuda.Event(enable_timing=True, external=True)
        stop = torch.cuda.Event(enable_timing=True, external=True)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream(dev)
            start.record(cs)
            stop.record(cs)
        g.replay()
        torch.cuda.synchronize(dev)
        head_start(stream)
        g.replay()
        torch.cuda.synchronize(dev)
        ts.append(start.elapsed_time(stop))
    return statistics.median(ts)


def finish_clocks(entries: list, sampler) -> None:
    """Replaces each entry's time window by the clock summary of its samples."""
    for e in entries:
        t0, t1 = e["clocks"]
        e["clocks"] = dict(sampler.summary(t0, t1), window="warm-up, both timed regions and a 0.3 s hold")


def sweep_points(qb, ops, dtypes, Ms, Ns, K, W, dev, stream, peak) -> list:
    """Every point of the M x N grid at K steps (graph and call by call); each
    record keeps the times of its timed regions for finish_sweep_clocks."""
    points = []
    for op in ops:
        for dtype in dtypes:
            code = qb.QK_F32 if dtype == "f32" else qb.QK_BF16
            for M in Ms:
                for N in Ns:
                    if N > qb.qk_max_row_elements(OP_CODES[op], code):
                        continue  # longer rows than this operator takes
                    ms, _, t = time_entry(qb, op, dtype, M, N, 1.0, K, W, dev, stream,
                                          seed=2000 + N, hold_s=0.0)
                    rec = {"op": op, "dtype": dtype, "M": M, "N": N, "steps": K,
                           "TBps": tbs_of(op, dtype, M, N, ms["graph"]),
                           "frac": tbs_of(op, dtype, M, N, ms["graph"]) * 1e3 / peak,
                           "frac_stream": tbs_of(op, dtype, M, N, ms["stream"]) * 1e3 / peak,
                           "ms": ms["graph"], "ms_stream": ms["stream"],
                           "plan": qb.qk_get_plan(OP_CODES[op], code, M, N), **t}
                    points.append(rec)
    return points


def finish_sweep_clocks(points: list, sampler, out=None) -> None:
    """Each point's clock samples: those within 0.15 s of its timed regions."""
    for p in points:
        p["clocks"] = sampler.summary(p.pop("t0") - 0.15, p.pop("t1") + 0.15)
        if out is not None:
            out.write(json.dumps(p) + "\n")


def sweep_summary(points: list, t_window, sampler) -> dict:
    """Per operator and dtype: min and median fraction of peak over N >= 4096,
    and the worst point; every point as [op, dtype, M, N, frac, frac call by
    call, median SM MHz of its samples]."""
    groups = {}
    for p in points:
        groups.setdefault(f"{p['op']}_{p['dtype']}", []).append(p)
    per = {}
    for key, ps in groups.items():
        ge = [p for p in ps if p["N"] >= 4096] or ps
        worst = min(ge, key=lambda p: p["frac"])
        per[key] = {"points": len(ps), "points_N_ge_4096": len(ge),
                    "min_frac_N_ge_4096": worst["frac"],
                    "median_frac_N_ge_4096": statistics.median(p["frac"] for p in ge),
                    "min_frac_stream_N_ge_4096": min(p["frac_stream"] for p in ge),
                    "median_frac_stream_N_ge_4096": statistics.median(p["frac_stream"] for p in ge),
                    "worst": {"M": worst["M"], "N": worst["N"], "frac": worst["frac"],
                              "TBps": worst["TBps"]}}
    ge_all = [p for p in points if p["N"] >= 4096]
    return {
        "grid": {"M": sorted({p["M"] for p in points}), "N": sorted({p["N"] for p in points}),
                 "ops": sorted({p["op"] for p in points}), "dtypes": sorted({p["dtype"] for p in points})},
        "launch": "cuda_graph (frac) and call by call (frac_stream)",
        "per_kernel": per,
        "points_N_ge_4096_at_or_above_0.85": sum(p["frac"] >= 0.85 for p in ge_all),
        "points_N_ge_4096": len(ge_all),
        "clocks": sampler.summary(*t_window),
        "points": [[p["op"], p["dtype"], p["M"], p["N"], round(p["frac"], 4), round(p["frac_stream"], 4),
                    p["clocks"]["sm_mhz"]] for p in points],
    }


def run_sweep(args, path):
    """Every point of the M x N sweep grid (--sweep-ops x fp32/bf16 x M x N),
    timed with the library's default plan, one JSON line per point into
    `path`; the summary line goes to stdout."""
    from memory_bound_row_rmsnorm_gb300 import binding as qb
    from memory_bound_row_rmsnorm_gb300 import build as qk_build
    qk_build.build()
    qb.load_library()
    torch.cuda.set_device(0)
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev)
    peak, peak_src = measured_peak()
    sweep_m = [int(v) for v in args.sweep_m.split(",")] if args.sweep_m else list(syn.SWEEP_M)
    sweep_n = [int(v) for v in args.sweep_n.split(",")] if args.sweep_n else list(syn.SWEEP_N)
    with ClockSampler(0) as sampler:
        t0 = time.time()
        points = sweep_points(qb, args.sweep_ops.split(","), ("f32", "bf16"), sweep_m, sweep_n,
                              args.steps, args.warmup, dev, stream, peak)
        t1 = time.time()
        time.sleep(0.3)  # let the sampler's last lines arrive
    with open(path, "w") as fout:
        finish_sweep_clocks(points, sampler, fout)
    summ = sweep_summary(points, (t0, t1), sampler)
    summ.pop("points")
    print(json.dumps({"sweep": path, "peak_gbs": peak, "peak_source": peak_src, **summ}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(ALL_WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--sweep", metavar="JSONL", help="time every sweep point instead; write them here")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="--impl reference: total CPU time budget of the timed steps")
    ap.add_argument("--sweep-ops", default="softmax,rmsnorm,xent",
                    help="operators of the sweep (also softmax_bwd, rmsnorm_bwd, xent_bwd, layernorm)")
    ap.add_argument("--sweep-m", help="comma-separated row counts of the sweep (default: the sweep grid)")
    ap.add_argument("--sweep-n", help="comma-separated row lengths of the sweep (default: the sweep grid)")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the per-workload block and the sweep summary of the default line")
    ap.add_argument("--rows", type=int, default=0,
                    help="run the workload with this many rows instead of its own M (small cases for "
                         "multi-metric profiler captures); the line then names the reduced shape")
    ap.add_argument("--hold", type=float, default=HOLD_S,
                    help="seconds of untimed steps after the timed regions (clock samples)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.sweep:
        run_sweep(args, args.sweep)
        return
    op, dtype, M, N, sigma = ALL_WORKLOADS[args.workload]
    if args.rows > 0:
        M = args.rows

    if args.impl == "reference":
        run_reference(args, op, dtype, M, N, sigma)
        return

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    else:
        torch.cuda.set_device(0)
    dev = torch.device(f"cuda:{local}")

    from memory_bound_row_rmsnorm_gb300 import binding as qb
    from memory_bound_row_rmsnorm_gb300 import build as qk_build
    if rank == 0 or ws == 1:
        qk_build.build()
    if ws > 1:
        dist.barrier()
    qb.load_library()
    peak, peak_src = measured_peak()
    sampler = ClockSampler(local).__enter__()

    # rotating input/output sets: > 4x L2 in total
    set_bytes = min_bytes(op, dtype, M, N)
    nsets = n_sets(set_bytes)
    sets = [make_set(op, dtype, M, N, sigma, rank_seed(rank, i), dev) for i in range(nsets)]
    stream = torch.cuda.current_stream(dev)
    code = qb.QK_F32 if dtype == "f32" else qb.QK_BF16
    plan = qb.qk_get_plan(OP_CODES[op], code, M, N)
    torch.cuda.synchronize(dev)

    t_start = time.time()
    for i in range(args.warmup):
        inp, out = sets[i % nsets]
        launch(qb, op, dtype, inp, out, M, N, stream)
    torch.cuda.synchronize(dev)
    if qb.qk_get_device_status(stream) != qb.QK_OK:
        raise RuntimeError("device status reports a failure after warm-up")

    K = args.steps
    elapsed = {}
    for mode in ("graph", "stream"):  # the same K steps, as one graph replay, then call by call
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        start, stop = timed_launches(qb, op, dtype, sets, M, N, K, stream, mode == "graph", dev)
        torch.cuda.synchronize(dev)
        if ws > 1:
            dist.barrier()
        ms = start.elapsed_time(stop)
        elapsed[mode] = max_over_ranks(ms, dist, dev) if ws > 1 else ms
    long_steps = None
    if elapsed["graph"] < LONG_REGION_MS:  # see LONG_REGION_MS
        long_steps = min(LONG_MAX_STEPS, max(K, math.ceil(LONG_TARGET_MS * K / elapsed["graph"])))
        if ws > 1:
            dist.barrier()
        start, stop = timed_launches(qb, op, dtype, sets, M, N, long_steps, stream, True, dev)
        torch.cuda.synchronize(dev)
        if ws > 1:
            dist.barrier()
        ms = start.elapsed_time(stop)
        elapsed["graph_long"] = max_over_ranks(ms, dist, dev) if ws > 1 else ms
    floor_ms = region_floor_ms(dev, stream)
    if args.hold > 0:
        hold(qb, op, dtype, sets, M, N, stream, dev, args.hold, elapsed["graph"] / K)
    t_end = time.time()
    status = qb.qk_get_device_status(stream)
    if status != qb.QK_OK:
        raise RuntimeError(f"device status: {qb.qk_status_string(status)}")

    elapsed_ms = elapsed["graph"]
    value = whole_job_tbs(set_bytes, ws, K, elapsed_ms)
    stream_value = whole_job_tbs(set_bytes, ws, K, elapsed["stream"])
    line_roofline = roofline(op, dtype, M, N, elapsed_ms / K, peak, peak_src,
                             recorded_traffic(args.workload, plan) if args.rows <= 0 else None)

    # ---- end to end: pinned host buffers, copies inside the timed region ----
    e2e_sets = sets[:2] if nsets >= 2 else sets + [make_set(op, dtype, M, N, sigma, rank_seed(rank, 1), dev)]
    e2e_ms, E, h2d, d2h = e2e_pipelined(qb, op, dtype, e2e_sets, M, N, max(3, args.e2e_steps), dev)
    if ws > 1:
        e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    e2e_value = whole_job_tbs(set_bytes, ws, E, e2e_ms)
    del sets, e2e_sets
    torch.cuda.empty_cache()

    if rank != 0:
        sampler.__exit__(None, None, None)
        if ws > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    per_workload, points, sweep_window = None, None, None
    if ws == 1 and not args.no_extras:
        per_workload = [workload_entry(qb, name, K, args.warmup, dev, stream, peak, peak_src)
                        for name in list(syn.WORKLOADS) + list(syn.BWD_WORKLOADS) + list(syn.NEXT_WORKLOADS)
                        if name != args.workload]
        t0 = time.time()
        points = sweep_points(qb, ("softmax", "rmsnorm", "xent"), ("f32", "bf16"), syn.SWEEP_M, syn.SWEEP_N,
                              K, args.warmup, dev, stream, peak)
        sweep_window = (t0, time.time())
    time.sleep(0.3)  # let the sampler's last lines arrive
    sampler.__exit__(None, None, None)
    clocks = sampler.summary(t_start, t_end)
    sweep = None
    if per_workload is not None:
        finish_clocks(per_workload, sampler)
        finish_sweep_clocks(points, sampler)
        sweep = sweep_summary(points, sweep_window, sampler)

    cpu = None
    if ws == 1 and args.cpu_seconds > 0:
        rate, cores, sample, _ = cpu_oracle_rate(op, dtype, M, N, sigma, args.cpu_seconds)
        one = cpu_single_core_rate(op, dtype, N, sigma, min(2.0, args.cpu_seconds / 5))
        cpu = {"value": rate, "unit": "TB/s", "cores": cores, "kind": "oracle", "sample": sample,
               "single_core_value": one, "cpu_model": cpu_model()}

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TB/s",
        "n_gpus": ws,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": elapsed_ms / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32" if dtype == "f32" else "bf16 in/out, f32 accumulate",
        "data": "synthetic",
        "config": {"workload": args.workload if args.rows <= 0 else f"{args.workload} at {M} rows",
                   "op": op, "M": M, "N": N, "input_dtype": dtype, "rows_per_gpu": M, "launch": "cuda_graph: the K calls captured once, replayed once",
                   "l2": f"{nsets} rotating input/output set(s) "
                   f"({nsets * set_bytes / 2**20:.0f} MiB) > 4x L2", "plan": plan},
        "stream": {"value": stream_value, "unit": "TB/s", "ms_per_step": elapsed["stream"] / K,
                   "frac": stream_value * 1e3 / ws / peak,
                   "how": "the same K steps issued call by call from Python, in their own timed region"},
        "roofline": line_roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "TB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": E,
                "how": "pinned host buffers; copy-in, call, copy-out every step, pipelined over 3 streams"},
        "gpu_launches": K * kernels_per_step(op),
        "clocks": dict(clocks, window="warm-up, both timed regions and a 0.3 s hold of the same steps"),
        "region_floor_us": floor_ms * 1e3,
    }
    if long_steps is not None:
        line["long_region"] = long_region_entry(op, dtype, M, N, long_steps,
                                                elapsed["graph_long"] / long_steps, peak)
        line["long_region"]["value"] *= ws
    if per_workload is not None:
        line["per_workload"] = per_workload
    if sweep is not None:
        line["sweep"] = sweep
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
