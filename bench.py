"""Benchmark of the fused cross-entropy hot path (and the row softmax) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gbce|reference]

One step is one ``ce_fwd_bwd`` call (target load, ignore test, non-ignored
count, online normaliser, in-place gradient, row losses, mean) over the
whole batch of the workload, inputs resident in HBM.  The call overwrites its
input, so before every step the pristine logits are copied back and L2 is
flushed (a 512 MB buffer written, then another read so that the written
lines are evicted before the timer starts), outside the timed span; each step
is timed alone with CUDA events between a barrier + synchronize on both
sides.  Rank 0 prints one JSON line.

With N > 1 (torchrun) every rank runs its own replica of the workload on its
own GPU (rows are independent; there is no collective on the data path) and
the value is the rows of all ranks over the slowest rank's time.

The line also carries ``workloads``: every configuration of the suite (the
CE workloads 64x1000 fp32, 8192x32000 bf16, 16384x128256 bf16, 4096x250007
fp32 and its 2-row all-ignored call; the fp32 softmax forward and backward at
4096 x N, N in {256, 1024, 4096, 16384}), each timed kernel-only with the same
restore, flush and CUDA-event method, with rows/s, algorithmic GB/s and the
fraction of the measured copy bandwidth.

``--impl reference`` times the CPU oracle (double precision, all host cores)
on a bounded sample of the same workload per step instead.
"""
import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "fused CE fwd+bwd rows/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
DEFAULT_WORKLOAD = "ce_bf16_16384x128256"
# the large-vocabulary CE workloads held to >= 80% of the measured copy bandwidth
GATED_CE = ("ce_bf16_8192x32000", "ce_bf16_16384x128256", "ce_f32_4096x250007")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # HBM3e nominal bandwidth of a GB300, reported beside the measured peak
E2E_STEPS = 20  # timed end-to-end steps (each moves 4.2 GB over the host link)
E2E_WARMUP = 3  # untimed end-to-end steps first (the first carries the one-time set-up)
L2_FLUSH_BYTES = 512 << 20  # > 2x the 129 MB L2
PROFILE_DIR = os.path.join(ROOT, "profiles")
KERNEL_SOURCES = [os.path.join(ROOT, "cross_entropy_loss_ce_gb300", "csrc", f)
                  for f in ("row_kernels.cuh", "device.cuh")]
BSR_KERNEL_SOURCES = [os.path.join(ROOT, "cross_entropy_loss_ce_gb300", "csrc", f)
                      for f in ("bsr_kernels.cuh", "device.cuh")]


# ---------------------------------------------------------------------------
# helpers

def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def esize(dtype):
    return 4 if dtype == torch.float32 else 2


def ce_algorithmic_bytes(w, targets_host: np.ndarray) -> int:
    """Bytes the method must move per launch of the row kernel: every live row
    read once and written once, every ignored row written once, plus per row
    the int64 target read and the fp32 row loss written."""
    ignored = int((targets_host == workloads.IGNORE_INDEX).sum())
    live = w.M - ignored
    row = w.V * esize(w.dtype)
    return live * 2 * row + ignored * row + w.M * (8 + 4)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(paths=KERNEL_SOURCES) -> str:
    """A digest of the kernel sources with comments and whitespace removed, so
    that a profile stays valid across edits that change no code."""
    h = hashlib.sha256()
    for p in paths:
        with open(p) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, prefix: str = "ce_rows", paths=KERNEL_SOURCES):
    """DRAM bytes per launch of a kernel from the committed ncu summary
    profiles/<prefix>_<workload>.txt, or None when there is none or the kernel
    source changed since."""
    path = os.path.join(PROFILE_DIR, f"{prefix}_{workload}.txt")
    try:
        text = open(path).read()
    except OSError:
        return None
    src = re.search(r"kernel_source_sha256_16:\s*(\w+)", text)
    val = re.search(r"dram_bytes_per_full_launch:\s*([0-9.eE+]+)", text)
    if not src or not val or src.group(1) != kernel_source_hash(paths):
        return None
    return float(val.group(1))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.reader.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def barrier_sync(ws):
    if ws > 1:
        torch.distributed.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def _collective_device():
    # NCCL reduces CUDA tensors; gloo (the CPU tests of this harness) host tensors
    return "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=_collective_device())
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=_collective_device())
    torch.distributed.all_reduce(t)
    return float(t.item())


def replica_throughput(rows_this_rank: float, ms_this_rank: float, ws: int):
    """(rows of all ranks / slowest rank's seconds, slowest rank's ms): the
    whole-job value of N independent replicas."""
    ms = max_over_ranks(ms_this_rank, ws)
    return sum_over_ranks(rows_this_rank, ws) / (ms / 1e3), ms


# ---------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, on this host's cores

def oracle_rows_per_s(w, x_host: torch.Tensor, t_host: torch.Tensor, block: int = 512,
                      min_seconds: float = 0.0, max_passes: int = 1, nthreads: int = 0):
    """Time the oracle (loss + full gradient) over the rows of x_host, in blocks;
    repeat the pass (up to max_passes) until min_seconds have elapsed.
    Returns (rows/s, seconds, threads, passes)."""
    import oracle
    V = w.V
    xa = oracle.host_array(x_host)
    ta = t_host.numpy()
    n, _ = oracle.ce_count(ta, V)
    nthreads = nthreads or oracle.default_threads()
    t0 = time.perf_counter()
    passes = 0
    while passes < max(max_passes, 1):
        for b0 in range(0, xa.shape[0], block):
            rows = np.arange(b0, min(b0 + block, xa.shape[0]))
            oracle.ce_rows(xa, ta, V, n, rows=rows, nthreads=nthreads)
        passes += 1
        if time.perf_counter() - t0 >= min_seconds:
            break
    dt = time.perf_counter() - t0
    return passes * xa.shape[0] / dt, dt, nthreads, passes


def single_core_oracle():
    """The oracle on one host core for the smallest CE workload (all 64 rows)
    and the 8192 x 32000 bf16 one (its first 1024 rows): rows/s each."""
    out = {}
    for name, rows in (("ce_f32_64x1000", 64), ("ce_bf16_8192x32000", 1024)):
        w = workloads.CE_WORKLOADS[name]
        x, t = workloads.make_ce_inputs(w.with_rows(rows), "cpu")
        rps, dt, _, passes = oracle_rows_per_s(w, x, t, min_seconds=0.5, max_passes=50,
                                               nthreads=1)
        out[name] = {"rows_per_s": rps, "rows": rows, "passes": passes, "seconds": dt}
    return out


def run_reference(args, ws, rank):
    """--impl reference: the oracle on the host cores, a bounded sample per step."""
    if rank != 0:
        return
    w = workloads.CE_WORKLOADS[args.workload]
    sample = args.ref_rows
    ws_ = w.with_rows(sample)
    x, t = workloads.make_ce_inputs(ws_, "cpu")
    for _ in range(args.warmup):
        oracle_rows_per_s(w, x, t)
    times = []
    threads = 1
    for _ in range(args.steps):
        _, dt, threads, _ = oracle_rows_per_s(w, x, t)
        times.append(dt)
    total = float(np.sum(times))
    value = sample * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name + (f" (first {w.M} rows)" if args.rows else ""), "M": w.M, "V": w.V, "logits_dtype": str(w.dtype),
                   "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": threads, "kind": "oracle",
                         "sample": f"{sample} rows of {w.name} per step (seeded CPU draw), "
                                   f"loss and full gradient in double precision"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the CUDA path

class L2Flush:
    """Between timed calls: write every line of a buffer larger than L2, then
    read a second such buffer.  The read evicts the first buffer's dirty lines,
    so their write-back happens here, untimed, instead of inside the next timed
    kernel (measured: up to 126 MB of write-back, +8 us on a 134 MB softmax),
    and the timed kernel starts with none of its inputs in L2."""

    def __init__(self, nbytes: int = L2_FLUSH_BYTES):
        self.w = torch.zeros(nbytes // 4, dtype=torch.float32, device="cuda")
        self.r = torch.ones(nbytes // 4, dtype=torch.float32, device="cuda")
        self.sink = torch.zeros((), dtype=torch.float32, device="cuda")


def flush_l2(f: L2Flush):
    f.w.add_(1)
    torch.sum(f.r, dim=0, out=f.sink)


def time_ce(w, xd0, td, steps, warmup, ws, flush):
    """(step ms summed over K steps, row-kernel ms per launch, loss, median step ms).

    Every step restores the pristine logits and flushes L2 (untimed), then
    one ce_fwd_bwd call sits between two CUDA events.  The K steps are
    enqueued back to back inside one barrier + synchronize bracket, so the
    host runs ahead and the events time the device work of the call alone.
    A second pass with the library's kernel events enabled gives the row
    kernel's own duration for the roofline."""
    import cross_entropy_loss_ce_gb300 as gbce
    xd = torch.empty_like(xd0)
    loss = torch.empty((), dtype=torch.float32, device="cuda")
    for _ in range(warmup):
        xd.copy_(xd0)
        gbce.ce_fwd_bwd(xd, td, workloads.IGNORE_INDEX, loss)
    torch.cuda.synchronize()
    if gbce.last_error() != gbce.OK:
        raise RuntimeError("device error flag raised during warm-up")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    stops = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    barrier_sync(ws)
    for i in range(steps):
        xd.copy_(xd0)
        flush_l2(flush)
        starts[i].record()
        gbce.ce_fwd_bwd(xd, td, workloads.IGNORE_INDEX, loss)
        stops[i].record()
    barrier_sync(ws)
    step_ms = sorted(a.elapsed_time(b) for a, b in zip(starts, stops))
    total = sum(step_ms)
    median = (step_ms[(steps - 1) // 2] + step_ms[steps // 2]) / 2
    loss_val = float(loss.item())
    # the row kernel alone (its events split the call, so they are a separate pass)
    kernel_steps = max(steps // 4, 5)
    gbce.timing_read()
    gbce.timing_enable(True)
    for _ in range(kernel_steps):
        xd.copy_(xd0)
        flush_l2(flush)
        gbce.ce_fwd_bwd(xd, td, workloads.IGNORE_INDEX, loss)
    torch.cuda.synchronize()
    kms, launches = gbce.timing_read()
    gbce.timing_enable(False)
    if gbce.last_error() != gbce.OK:
        raise RuntimeError("device error flag raised during the timed steps")
    return total, kms / max(launches, 1), loss_val, median


def time_ce_e2e(w, x_pinned, t_pinned, steps, ws):
    """End to end through the public host-buffer call ce_fwd_bwd_host: pinned
    host -> device copies of the step's targets and logits (the logits in row
    chunks that overlap the row kernels), the call, the loss read back into
    pinned host memory."""
    import cross_entropy_loss_ce_gb300 as gbce
    grad = torch.empty(x_pinned.shape, dtype=x_pinned.dtype, device="cuda")
    loss_host = torch.empty((), dtype=torch.float32).pin_memory()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_ms = []
    for i in range(E2E_WARMUP + steps):
        barrier_sync(ws)
        start.record()
        gbce.ce_fwd_bwd_host(x_pinned, t_pinned, workloads.IGNORE_INDEX, grad, loss_host)
        stop.record()
        barrier_sync(ws)
        if i >= E2E_WARMUP:
            step_ms.append(start.elapsed_time(stop))
    h2d = x_pinned.numel() * x_pinned.element_size() + t_pinned.numel() * 8
    return sum(step_ms), h2d, 4, step_ms


def host_link_gbs(x_pinned, reps: int = 3) -> float:
    """Host -> device bandwidth of one plain copy of the pinned logits, measured
    in the same run (context for the e2e figure: the link bounds it)."""
    dst = torch.empty(x_pinned.shape, dtype=x_pinned.dtype, device="cuda")
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = float("inf")
    for _ in range(reps):
        torch.cuda.synchronize()
        start.record()
        dst.copy_(x_pinned, non_blocking=True)
        stop.record()
        torch.cuda.synchronize()
        best = min(best, start.elapsed_time(stop))
    del dst
    return x_pinned.numel() * x_pinned.element_size() / (best / 1e3) / 1e9


def kernel_ms(call, steps, warmup, flush, ws=1, restore=None):
    """Mean duration of the library's row kernel in `call` (CUDA events the
    library records around it on the call's stream), over `steps` calls, each
    preceded (untimed) by `restore` and an L2 flush; max over ranks.  The calls
    are enqueued back to back between one barrier + synchronize on each side:
    a synchronize between a flush and its call would let the start event fire
    before the host has even enqueued the kernel, timing the launch overhead
    of short kernels too."""
    import cross_entropy_loss_ce_gb300 as gbce
    for _ in range(warmup):
        if restore:
            restore()
        call()
    torch.cuda.synchronize()
    if gbce.last_error() != gbce.OK:
        raise RuntimeError("device error flag raised during warm-up")
    gbce.timing_read()
    gbce.timing_enable(True)
    barrier_sync(ws)
    for _ in range(steps):
        if restore:
            restore()
        flush_l2(flush)
        call()
    barrier_sync(ws)
    ms, n = gbce.timing_read()
    gbce.timing_enable(False)
    if gbce.last_error() != gbce.OK:
        raise RuntimeError("device error flag raised during the timed calls")
    return max_over_ranks(ms / max(n, 1), ws)


def softmax_traffic(direction: str, M: int, N: int):
    """DRAM bytes per launch of the softmax row kernel from its committed ncu
    summary, or None (no summary, or the kernel changed since)."""
    return profiled_traffic(f"f32_{M}x{N}", f"softmax_{direction}")


def entry(workload, kernel, ms, rows, alg_bytes, peak, traffic=None, gated=False, **extra):
    d = {"workload": workload, "kernel": kernel, "kernel_ms": ms,
         "rows_per_s": rows / (ms / 1e3), "algorithmic_bytes": alg_bytes,
         "gbs": alg_bytes / (ms / 1e3) / 1e9, "frac": alg_bytes / (ms / 1e3) / 1e9 / peak,
         "traffic": traffic, "gated": gated}
    d.update(extra)
    return d


def ce_workload_entry(w, xd0, td, steps, warmup, flush, peak, ws=1):
    """One CE workload through ce_fwd_bwd, kernel-only: the row kernel's time,
    the call's loss checked finite (NaN when every row is ignored)."""
    import cross_entropy_loss_ce_gb300 as gbce
    xd = torch.empty_like(xd0)
    loss = torch.empty((), dtype=torch.float32, device="cuda")
    ms = kernel_ms(lambda: gbce.ce_fwd_bwd(xd, td, workloads.IGNORE_INDEX, loss), steps, warmup,
                   flush, ws, restore=lambda: xd.copy_(xd0))
    t_host = td.cpu().numpy()
    alg = ce_algorithmic_bytes(w, t_host)
    kernel, C = gbce.plan("ce", w.M, w.V, w.dtype)
    all_ignored = bool((t_host == workloads.IGNORE_INDEX).all())
    lv = float(loss.item())
    if all_ignored != (lv != lv):
        raise RuntimeError(f"{w.name}: unexpected loss {lv}")
    named = workloads.CE_WORKLOADS.get(w.name)
    full = named is not None and w.M == named.M
    gated = w.name in GATED_CE and full and not all_ignored
    name = w.name if full else f"{w.name} (first {w.M} rows" + (", all ignored)" if all_ignored
                                                                  else ")")
    return entry(name, f"{kernel}<CE>" + (f", cluster of {C}" if C > 1 else ""), ms, w.M, alg,
                 peak, profiled_traffic(w.name) if full else None, gated, loss=lv)


def softmax_entries(N, steps, warmup, flush, peak, ws=1, M=workloads.SOFTMAX_M):
    """Softmax forward, then backward, on the M x N fp32 workload (M = 4096)."""
    import cross_entropy_loss_ce_gb300 as gbce
    x, y, dy = workloads.make_softmax_inputs(M, N, device="cuda")
    out = []
    yo, dx = torch.empty_like(x), torch.empty_like(x)
    for direction, call, nbytes, op in (
            ("fwd", lambda: gbce.softmax_fwd(x, yo), 2 * M * N * 4, "softmax_fwd"),
            ("bwd", lambda: gbce.softmax_bwd(y, dy, dx), 3 * M * N * 4, "softmax_bwd")):
        ms = kernel_ms(call, steps, warmup, flush, ws)
        kernel, C = gbce.plan(op, M, N, torch.float32)
        out.append(entry(f"softmax_{direction}_f32_{M}x{N}",
                         f"{kernel}<{op}>" + (f", cluster of {C}" if C > 1 else ""), ms, M,
                         nbytes, peak, softmax_traffic(direction, M, N), N >= 4096))
    del x, y, dy, yo, dx
    return out


SMALL_BATCH = 8  # rows of the small-batch CE entry


def all_workloads(steps, warmup, flush, peak, ws=1, c4=None):
    """Every configuration of the benchmark suite, kernel-only, one entry each:
    the CE workloads (64x1000 fp32, 8192x32000 bf16, 16384x128256 bf16,
    4096x250007 fp32 and its 2-row all-ignored call) and the fp32 softmax
    forward and backward at 4096 x N, N in {256, 1024, 4096, 16384}; then two
    small batches: the first 8 rows of the 16384x128256 workload and a one-row
    fp32 softmax of N = 128256.  Inputs are drawn on the device.  `c4`: the
    16384x128256 inputs when already resident.
    A last pair of entries times a one-row softmax (1 KB): the fixed cost of a
    launch between the two events, which bounds the small shapes."""
    out = []
    for w in workloads.CE_WORKLOADS.values():
        if c4 is not None and w.name == DEFAULT_WORKLOAD:
            xd0, td = c4
        else:
            xd0, td = workloads.make_ce_inputs(w, "cuda")
        out.append(ce_workload_entry(w, xd0, td, steps, warmup, flush, peak, ws))
        if w.name == "ce_f32_4096x250007":
            w2 = w.with_rows(2)
            t2 = torch.full((2,), workloads.IGNORE_INDEX, dtype=torch.int64, device="cuda")
            out.append(ce_workload_entry(w2, xd0[:2].clone(), t2, steps, warmup, flush, peak,
                                         ws))
        del xd0, td
        torch.cuda.empty_cache()
    for N in workloads.SOFTMAX_NS:
        out.extend(softmax_entries(N, steps, warmup, flush, peak, ws))
        torch.cuda.empty_cache()
    # small batches of long rows (each row split across a cluster): the first 8
    # rows of the 128256-column bf16 workload, and one fp32 softmax row of 128256
    w = workloads.CE_WORKLOADS[DEFAULT_WORKLOAD]
    if c4 is not None:
        x8, t8 = c4[0][:SMALL_BATCH].clone(), c4[1][:SMALL_BATCH].clone()
    else:
        x8, t8 = workloads.make_ce_inputs(w.with_rows(SMALL_BATCH), "cuda")
    out.append(ce_workload_entry(w.with_rows(SMALL_BATCH), x8, t8, steps, warmup, flush, peak, ws))
    del x8, t8
    out.extend(softmax_entries(128256, steps, warmup, flush, peak, ws, M=1))
    # the fixed cost of one launch between the events: a one-row softmax of 1 KB
    for e in softmax_entries(256, steps, warmup, flush, peak, ws, M=1):
        e["workload"] = "launch floor: " + e["workload"]
        out.append(e)
    return out


def bsr_algorithmic_bytes(meta, Z, es, lut_len) -> int:
    """Two reads (y, dy) and one write (dx) of every stored element, plus the table."""
    return 3 * Z * meta["nblocks"] * meta["block"] ** 2 * es + 4 * lut_len


def time_bsr(steps, warmup, ws, flush, peak, heads=0):
    """Block-sparse softmax backward on each block-sparse workload (dx out of
    place, so every step sees the same inputs): kernel time from the library's
    events, L2 flushed before each call.  ``heads`` > 0 keeps that many heads
    of each workload (a smaller case for profiling)."""
    import cross_entropy_loss_ce_gb300 as gbce
    out = []
    for w in workloads.BSR_WORKLOADS.values():
        if heads:
            w = w.with_sizes(H=heads)
        y, dy, lut, meta = workloads.make_bsr_inputs(w, device="cuda")
        dx = torch.empty_like(dy)
        call = lambda: gbce.softmax_bwd_bsr(y, dy, lut, meta["n_block_rows"], meta["nblocks"],
                                            meta["block"], meta["sizemax"], 1.0, dx)
        ms = kernel_ms(call, steps, warmup, flush, ws)
        b = bsr_algorithmic_bytes(meta, w.Z, esize(w.dtype), lut.numel())
        rows = w.Z * meta["n_block_rows"] * meta["block"]
        kernel, R = gbce.bsr_plan(meta["block"], meta["sizemax"], w.dtype)
        out.append({"workload": w.name + (f" ({heads} heads)" if heads else ""),
                    "kernel": kernel, "rows_per_slab_longest": R,
                    "timing": "kernel, CUDA events", "kernel_ms": ms,
                    "rows_per_s": rows / (ms / 1e3), "algorithmic_bytes": b,
                    "gbs": b / (ms / 1e3) / 1e9, "frac": b / (ms / 1e3) / 1e9 / peak,
                    "traffic": None if heads else profiled_traffic(
                        w.name, "softmax_bwd_bsr", BSR_KERNEL_SOURCES)})
        del y, dy, dx
        torch.cuda.empty_cache()
    return out


def run_gbce(args, ws, rank, local):
    import cross_entropy_loss_ce_gb300 as gbce
    gbce.load_library()
    torch.cuda.set_device(local)
    w = workloads.CE_WORKLOADS[args.workload]
    if args.rows:
        w = w.with_rows(args.rows)
    xd0, td = workloads.make_ce_inputs(w, "cuda")
    t_host = td.cpu().numpy()
    flush = L2Flush()
    peak, peak_kind = measured_peaks()

    with ClockSampler(local) as clocks:
        total_ms, kavg_ms, loss_val, median_ms = time_ce(w, xd0, td, args.steps, args.warmup, ws,
                                                         flush)
    clk = clocks.summary()
    value, total_ms = replica_throughput(float(w.M * args.steps), total_ms, ws)
    ms_per_step = total_ms / args.steps
    alg = ce_algorithmic_bytes(w, t_host)
    kavg_ms = max_over_ranks(kavg_ms, ws)
    achieved = alg / (kavg_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": profiled_traffic(w.name),
                "kernel": gbce.plan("ce", w.M, w.V, w.dtype)[0] + "<CE>", "kernel_ms": kavg_ms,
                "algorithmic_bytes": alg, "peak_kind": f"{peak_kind} (hbm_gbs, burst)",
                "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": achieved / NOMINAL_HBM_GBS}

    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step,
        "ms_per_step_median": max_over_ranks(median_ms, ws), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == torch.bfloat16 else "f32", "data": "synthetic",
        "config": {"workload": w.name + (f" (first {w.M} rows)" if args.rows else ""), "M": w.M, "V": w.V, "ignore_frac": w.ignore_frac,
                   "logits": f"N(0,{w.std}^2)" + (f" + {w.spike} spike/row" if w.spike else ""),
                   "l2": "inputs (4.2 GB) larger than L2, and before each step (untimed) a "
                         "512 MB buffer written, then another 512 MB read",
                   "parallelism": "replicas" if ws > 1 else "single GPU"},
        "step_hbm_gbs": alg / (ms_per_step / 1e3) / 1e9,
        "loss": loss_val,
        "roofline": roofline,
        "gpu_launches": 3 * args.steps,  # count, row and mean kernels
        "clocks": clk,
    }

    if not args.no_e2e:
        # before the per-workload timings: their multi-GB allocations and frees
        # measurably slow this process's later host-to-device copies
        x_pinned = xd0.cpu().pin_memory()
        t_pinned = td.cpu().pin_memory()
        e2e_steps = min(args.steps, E2E_STEPS)
        link_before = host_link_gbs(x_pinned)
        e2e_ms, h2d, d2h, step_ms = time_ce_e2e(w, x_pinned, t_pinned, e2e_steps, ws)
        link_after = host_link_gbs(x_pinned)
        e2e_ms = max_over_ranks(e2e_ms, ws)
        # the value is the mean over the steps; the spread and the link measured
        # on either side show a step slowed by other traffic on the host link
        ordered = sorted(step_ms)
        line["e2e"] = {"value": sum_over_ranks(float(w.M * e2e_steps), ws) / (e2e_ms / 1e3),
                       "unit": "rows/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": e2e_ms / e2e_steps,
                       "ms_per_step_median": ordered[len(ordered) // 2],
                       "ms_per_step_min": ordered[0], "ms_per_step_max": ordered[-1],
                       "ms_steps": [round(t, 2) for t in step_ms],
                       "host_link_h2d_gbs": min(link_before, link_after),
                       "host_link_h2d_gbs_before_after": [link_before, link_after]}
        del x_pinned

    if not args.no_workloads:
        # every configuration, kernel-only, with the same restore, flush and events
        line["workloads"] = all_workloads(max(args.steps // 5, 10), args.warmup, flush, peak, ws,
                                          c4=(xd0, td) if w.name == DEFAULT_WORKLOAD and
                                          not args.rows else None)

    if not args.no_softmax:
        line["softmax_bsr"] = time_bsr(max(args.steps // 2, 5), args.warmup, ws, flush, peak)

    if rank == 0 and not args.no_cpu_baseline:
        sample = min(args.cpu_rows, w.M)
        x_host = xd0[:sample].cpu()
        rps, dt, cores, passes = oracle_rows_per_s(w, x_host, td[:sample].cpu(),
                                                   min_seconds=10.0, max_passes=20)
        line["cpu_baseline"] = {"value": rps, "unit": "rows/s", "cores": cores, "kind": "oracle",
                                "sample": f"first {sample} rows of {w.name}, {passes} passes: "
                                          f"loss and full gradient in double precision, "
                                          f"{dt:.1f} s",
                                "single_core": single_core_oracle()}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_table(args, local):
    """--table: kernel-only time of every workload (one JSON line per entry)."""
    import cross_entropy_loss_ce_gb300 as gbce
    gbce.load_library()
    torch.cuda.set_device(local)
    peak, _ = measured_peaks()
    flush = L2Flush()
    steps = max(args.steps // 4, 10)
    for r in all_workloads(steps, args.warmup, flush, peak):
        print(json.dumps({"table": r["workload"], "kernel_us": 1e3 * r["kernel_ms"],
                          "rows_per_s": r["rows_per_s"], "alg_gbs": r["gbs"],
                          "frac_of_measured_peak": r["frac"], "kernel": r["kernel"]}),
              flush=True)
    for r in time_bsr(steps, args.warmup, 1, flush, peak):
        print(json.dumps({"table": r["workload"], "kernel_us": 1e3 * r["kernel_ms"],
                          "rows_per_s": r["rows_per_s"], "alg_gbs": r["gbs"],
                          "frac_of_measured_peak": r["frac"], "kernel": r["kernel"],
                          "rows_per_slab_longest": r["rows_per_slab_longest"]}), flush=True)


def run_only(args, local):
    """--only NAME: one workload kernel-only (a CE workload, or softmax_f32_4096xN
    for the forward and backward), its first --rows rows when given; one JSON
    line per entry.  A small, single-workload command for profiling."""
    import cross_entropy_loss_ce_gb300 as gbce
    gbce.load_library()
    torch.cuda.set_device(local)
    peak, _ = measured_peaks()
    flush = L2Flush()
    steps = max(args.steps, 1)
    if args.only in workloads.CE_WORKLOADS:
        w = workloads.CE_WORKLOADS[args.only]
        if args.rows:
            w = w.with_rows(args.rows)
        xd0, td = workloads.make_ce_inputs(w, "cuda")
        out = [ce_workload_entry(w, xd0, td, steps, args.warmup, flush, peak)]
    else:
        m = re.fullmatch(r"softmax_f32_(\d+)x(\d+)", args.only)
        if not m:
            raise SystemExit(f"--only: unknown workload {args.only!r}")
        out = softmax_entries(int(m.group(2)), steps, args.warmup, flush, peak,
                              M=args.rows or int(m.group(1)))
    for r in out:
        print(json.dumps(r), flush=True)


def run_bsr(args, local):
    """--bsr: kernel-only time of the block-sparse softmax backward workloads
    (one JSON line per workload)."""
    import cross_entropy_loss_ce_gb300 as gbce
    gbce.load_library()
    torch.cuda.set_device(local)
    peak, _ = measured_peaks()
    flush = L2Flush()
    for r in time_bsr(args.steps, args.warmup, 1, flush, peak, args.bsr_heads):
        print(json.dumps(r), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gbce", "reference"], default="gbce")
    ap.add_argument("--workload", choices=list(workloads.CE_WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--rows", type=int, default=0,
                    help="run the first ROWS rows of the workload only (profiling a small case)")
    ap.add_argument("--cpu-rows", type=int, default=16384)
    ap.add_argument("--ref-rows", type=int, default=256)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-softmax", action="store_true",
                    help="skip the block-sparse softmax backward timings")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-workload kernel timings (every CE and softmax config)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--bsr", action="store_true",
                    help="time only the block-sparse softmax backward workloads")
    ap.add_argument("--bsr-heads", type=int, default=0,
                    help="with --bsr: keep this many heads of each workload (profiling)")
    ap.add_argument("--table", action="store_true",
                    help="print the kernel time of every workload instead of the benchmark line")
    ap.add_argument("--only", default=None,
                    help="time one workload only: a CE workload name or softmax_f32_4096xN "
                         "(with --rows: its first ROWS rows); for profiling")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    ws, rank, local = dist_info()
    if ws > 1:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        torch.distributed.init_process_group(backend)
    try:
        if args.impl == "reference":
            run_reference(args, ws, rank)
        elif args.table:
            run_table(args, local)
        elif args.only:
            run_only(args, local)
        elif args.bsr:
            run_bsr(args, local)
        else:
            run_gbce(args, ws, rank, local)
    finally:
        if ws > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
