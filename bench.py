"""Benchmark of the LLM.int8() matmul (int8_matmul) on B300.

One step = one int8_matmul over one batch: the column-statistics pass, the row quantize +
outlier gather pass and the tensor-core matmul, on the FFN up-projection of a 13B-class
model (X fp16 [4096, 5120] with 0.2% outlier columns, W [20480, 5120], threshold 6.0), the
largest T x d -> 4d configuration that fits one GPU.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

N > 1 runs under torch.distributed (one process per GPU, NCCL): every rank multiplies its
own independent batch (weak scaling, no collective on the data path); the timed region
is bracketed by a barrier and a device synchronize, and the time is the max over ranks.
The reference arm (`--impl reference`) is the CPU oracle on the host cores, timed on a
bounded sample of rows of the same workload.

Prints one JSON line (rank 0). `--all` prints one line per configuration, the 6.7B line
with zeropoint activation codes (`--zeropoint`), the FFN block line (`--ffn` alone prints
only that one) and the standalone row quantizers.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "int8_matmul TOPS and % of INT8-tensor/HBM roofline on T×d→4d FFN GEMM"
UNIT = "TOPS"
DEFAULT_WORKLOAD = "ffn_13b_up"
ALL_CONFIGS = ["ffn_6.7b_up", "ffn_13b_up", "ffn_13b_down", "decode_176b_t1", "decode_176b_t8",
               "decode_176b_t64", "sweep_f0_thr6", "sweep_f0.1_thr6", "sweep_f0.5_thr6",
               "sweep_f2_thr6", "sweep_f0_thrinf", "sweep_f2_thrinf"]
FFN_METRIC = ("int8_ffn TOPS on the FFN block (X W_up^T -> ReLU -> W_down^T, LLM.int8() "
              "in both)")
DEFAULT_FFN = "ffn_13b_block"
L2_FLUSH_BYTES = 256 << 20
PEAKS_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def load_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        return json.load(open(path)), "measured"
    except (OSError, ValueError):
        return dict(PEAKS_FALLBACK), "fallback"


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
CSRC = os.path.join(ROOT, "int8_mixed_precision_03_b300", "csrc")
KERNEL_SOURCES = {
    "i8_gemm_kernel": ("gemm_i8.cu", "gemm_common.cuh", "sm103_ptx.cuh", "int8mm_internal.h"),
    "gemv_i8_kernel": ("gemv_i8.cu", "int8mm_internal.h"),
    "gemv_mma_kernel": ("gemv_mma.cu", "int8mm_internal.h"),
}
# decode-size kernels (the library's rule): T <= 8 on dp4a with the int8 codes in shared
# memory, 9 <= T <= 16 on mma.sync with 128-byte-padded code rows
GEMV_MAX_T, GEMV_MMA_MIN_T, GEMV_MAX_SMEM = 16, 9, 200 * 1024


def uses_gemv(w: synth.Workload) -> bool:
    if w.T < 1 or w.T > GEMV_MAX_T:
        return False
    if w.T >= GEMV_MMA_MIN_T:
        xs = (w.d_in + 127) // 128 * 128 + 64
        return w.T * xs <= GEMV_MAX_SMEM
    return w.T * w.d_in <= GEMV_MAX_SMEM


def matmul_kernel(w: synth.Workload) -> str:
    if not uses_gemv(w):
        return "i8_gemm_kernel"
    return "gemv_mma_kernel" if w.T >= GEMV_MMA_MIN_T else "gemv_i8_kernel"


def kernel_source_hash(kernel: str) -> str:
    """sha256 of the kernel's sources with comments and blank lines removed, so that a
    change of wording in a comment keeps the counters taken on the same code."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        src = open(os.path.join(CSRC, f), encoding="utf-8").read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        lines = [ln.rstrip() for ln in src.splitlines() if ln.strip()]
        h.update("\n".join(lines).encode())
    return h.hexdigest()


def measured_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of the matmul kernel from the committed ncu capture, if it was
    taken on this exact kernel source and workload; None otherwise."""
    try:
        rec = json.load(open(TRAFFIC_FILE)).get(workload)
    except (OSError, ValueError, AttributeError):
        return None
    if not rec or rec.get("kernel") != kernel or rec.get("source_sha256") != kernel_source_hash(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


def workload_ops(w: synth.Workload) -> float:
    """Algorithmic int8 operations of one matmul: 2 * T * d_in * d_out."""
    return 2.0 * w.T * w.d_in * w.d_out


def algorithmic_bytes(w: synth.Workload) -> int:
    """Minimum bytes the method must move: X, CB, SCB, bias, Y."""
    return 2 * w.T * w.d_in + w.d_in * w.d_out + 4 * w.d_out + 2 * w.d_out + 2 * w.T * w.d_out


def matmul_bytes(w: synth.Workload) -> int:
    """Algorithmic bytes of the matmul kernel: CB, the activation codes (int8 for the
    decode kernel, fp16 for the tensor-core kernel), SCB, rowabs, bias and Y (the outlier
    slices are a few KB and are left out)."""
    code_bytes = 1 if uses_gemv(w) else 2
    return (w.d_in * w.d_out + code_bytes * w.T * w.d_in + 4 * w.d_out + 4 * w.T
            + 2 * w.d_out + 2 * w.T * w.d_out)


def hbm_bound(w: synth.Workload) -> bool:
    """Decode shapes (T <= 64): streaming CB from HBM takes longer than the arithmetic."""
    return w.T <= 64


def roofline(w: synth.Workload, matmul_ms: float, peaks: dict, peak_src: str,
             zeropoint: bool = False) -> dict:
    """Roofline of the dominant kernel (the matmul), from its CUDA-event time."""
    s = matmul_ms / 1e3
    kernel = "i8_gemm_kernel" if zeropoint else matmul_kernel(w)
    traffic = None if zeropoint else measured_traffic(w.name, kernel)
    if hbm_bound(w):
        achieved = matmul_bytes(w) / s / 1e9
        peak = float(peaks["hbm_gbs"])
        desc = {"gemv_i8_kernel": "gemv_i8_kernel (dp4a on CUDA cores, int8 codes)",
                "gemv_mma_kernel": "gemv_mma_kernel (mma.sync m16n8k16 fp16 on exact int8 codes)",
                "i8_gemm_kernel": "i8_gemm_kernel (tcgen05 kind::f16 on exact int8 codes), "
                                  "decode tile"}[kernel]
        return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic,
                "algorithmic_bytes": matmul_bytes(w), "kernel": desc,
                "peak_source": f"hbm_gbs, {peak_src} (MEASURED_PEAKS.json)"}
    achieved = workload_ops(w) / s / 1e12
    peak = float(peaks["bf16_tflops"])
    return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "traffic": traffic,
            "kernel": "i8_gemm_kernel (tcgen05 kind::f16 on exact int8 codes)",
            "peak_source": f"bf16_tflops burst, {peak_src} (MEASURED_PEAKS.json); the int8 "
                           "product runs on kind::f16, at the bf16/fp16 rate"}


# ------------------------------------------------------------------ timing helpers
L2_NOTE = ("flushed between timed steps: 256 MiB written, then another 256 MiB read, so that "
           "each timed step starts from a cold L2 holding no dirty lines (untimed)")


class L2Flush:
    """L2 flush between timed steps. Writing a buffer larger than L2 evicts everything, but
    leaves L2 full of dirty lines whose write-back would then compete with the timed kernels
    for DRAM; reading a second buffer of the same size afterwards writes them back before
    the timed step starts."""

    def __init__(self, device):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device)

    def __call__(self, k: int) -> None:
        import torch
        self.w.fill_(k & 0xff)
        torch.amax(self.r)


def event_time_us(fn, flush, n: int = 20, warm: int = 3) -> float:
    """Mean CUDA-event time of fn() in microseconds, L2 flushed before each call."""
    import torch
    out = []
    for k in range(n + warm):
        flush(k)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        if k >= warm:
            out.append((a, b))
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in out) * 1e3


# ------------------------------------------------------------------ distributed plumbing
def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def aggregate(elapsed_s: float, units: float, group=None) -> tuple[float, float]:
    """(max elapsed over ranks, total units over ranks). Works for any backend."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return elapsed_s, units
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(u.item())


# ------------------------------------------------------------------ clocks
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons; only the samples taken inside
    the timed region (between mark_start() and mark_end(), host wall clock) are kept."""

    def __init__(self, gpu_index: int):
        self.proc = None
        self.t0 = self.t1 = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu=timestamp,{CLOCK_QUERY}",
                 "--format=csv,noheader,nounits", "-i", str(gpu_index), "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)   # let the sampler start before the timed region opens
        except OSError:
            self.proc = None

    def mark_start(self) -> None:
        self.t0 = time.time()

    def mark_end(self) -> None:
        self.t1 = time.time()

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        import datetime
        sm, mx, reasons, total = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            total += 1
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm_v, mx_v = float(f[2]), float(f[3])
            except ValueError:
                continue
            if self.t0 is not None and not (self.t0 <= ts <= (self.t1 or ts)):
                continue
            sm.append(sm_v)
            mx.append(mx_v)
            for n, v in zip(names, f[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": f"no sample fell inside the timed region ({total} taken)"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ oracle (CPU) arm
def oracle_matmul(zeropoint: bool):
    """The oracle's matmul: absmax codes, or the zeropoint variant."""
    import oracle
    return oracle.int8_matmul_zeropoint if zeropoint else oracle.int8_matmul


def calibrated_rows(w, X, CBo, SCBo, bias, nthreads: int, seconds: float,
                    zeropoint: bool = False) -> int:
    """Rows of X whose oracle evaluation takes about `seconds` on these host cores: the
    per-row cost is the slope between two timed samples (the fixed cost of a call, the
    outlier scan over all of X, cancels)."""
    fn = oracle_matmul(zeropoint)

    def timed(n):
        rows = np.linspace(0, w.T - 1, n).astype(np.int64)
        t0 = time.perf_counter()
        fn(X, CBo, SCBo, w.threshold, bias, rows=rows, nthreads=nthreads, want_acc=False)
        return time.perf_counter() - t0

    n1, n2 = min(w.T, 4 * nthreads), min(w.T, 16 * nthreads)
    t1, t2 = timed(n1), timed(n2)
    per_row = max((t2 - t1) / max(n2 - n1, 1), t2 / n2 * 0.25, 1e-7)
    fixed = max(t2 - per_row * n2, 0.0)
    return int(min(w.T, max(1, round((seconds - fixed) / per_row))))


def cpu_baseline_sample(w, X, CBo, SCBo, bias, nthreads: int, seconds: float = 15.0,
                        zeropoint: bool = False) -> dict:
    """The oracle as it stands, timed on a bounded sample of rows of the workload."""
    fn = oracle_matmul(zeropoint)
    rows_n = calibrated_rows(w, X, CBo, SCBo, bias, nthreads, seconds, zeropoint)
    rows = np.linspace(0, w.T - 1, rows_n).astype(np.int64)
    reps, t0 = 0, time.perf_counter()
    while True:   # the whole workload may take less than `seconds`: repeat it
        fn(X, CBo, SCBo, w.threshold, bias, rows=rows, nthreads=nthreads, want_acc=False)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= 0.6 * seconds:
            break
    ops = 2.0 * rows_n * w.d_in * w.d_out * reps
    codes = "zeropoint" if zeropoint else "absmax"
    return {"value": ops / dt / 1e12, "unit": UNIT, "cores": nthreads, "kind": "oracle",
            "sample": f"{reps} x {rows_n} of {w.T} rows of {w.name} (each pass: outlier scan "
                      f"of all of X, then {codes} quantize, int8 product, fp16 outlier product "
                      f"and bias for those rows), {dt:.1f} s wall"}


def ffn_cpu_baseline(f, blk, nthreads: int, seconds: float = 15.0) -> dict:
    """The oracle's FFN block as it stands on the first rows of X (a smaller batch of the
    same block: the down projection's outlier columns need every row of its input, so the
    sample is a batch, not a row subset), sized to about `seconds`, scaled to TOPS."""
    import oracle
    CBu, SCBu = oracle.quantize_weight(blk["W_up"])
    CBd, SCBd = oracle.quantize_weight(blk["W_down"])

    def run(n):
        t0 = time.perf_counter()
        oracle.ffn(blk["X"][:n], CBu, SCBu, CBd, SCBd, f.threshold, blk["b_up"], blk["b_down"],
                   "relu", nthreads=nthreads)
        return time.perf_counter() - t0

    n1 = min(f.T, 2 * nthreads)
    t1 = run(n1)
    n = int(min(f.T, max(n1, round(n1 * seconds / max(t1, 1e-3)))))
    dt = run(n) if n != n1 else t1
    return {"value": 4.0 * n * f.d_model * f.d_ff / dt / 1e12, "unit": UNIT,
            "cores": nthreads, "kind": "oracle",
            "sample": f"the first {n} of {f.T} tokens of {f.name} through the whole block "
                      f"(both outlier scans, quantize, int8 products, ReLU), {dt:.1f} s wall"}


def run_reference(args) -> None:
    """The oracle as it stands, on the host cores, one bounded sample per step."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    w = synth.WORKLOADS[args.workload]
    X, W, bias = synth.make_x(w), synth.make_w(w), synth.make_bias(w)
    CBo, SCBo = oracle.quantize_weight(W)
    nthreads = os.cpu_count() or 1
    # each step a bounded sample: the whole warm-up + timed run takes about two minutes
    per_step = args.ref_budget_s / max(1, args.steps + args.warmup)
    rows_n = calibrated_rows(w, X, CBo, SCBo, bias, nthreads, per_step)
    rows = np.linspace(0, w.T - 1, rows_n).astype(np.int64)
    for _ in range(args.warmup):
        oracle.int8_matmul(X, CBo, SCBo, w.threshold, bias, rows=rows, nthreads=nthreads,
                           want_acc=False)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.int8_matmul(X, CBo, SCBo, w.threshold, bias, rows=rows, nthreads=nthreads,
                           want_acc=False)
    dt = time.perf_counter() - t0
    ops = 2.0 * rows_n * w.d_in * w.d_out * args.steps
    value = ops / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "s8",
        "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "d_in": w.d_in, "d_out": w.d_out,
                   "threshold": w.threshold, "n_outlier_cols": w.n_outlier_cols,
                   "sample_rows": rows_n},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": nthreads, "kind": "oracle",
                         "sample": f"{rows_n} of {w.T} rows per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm
def run_ours(args) -> None:
    import torch
    import torch.distributed as dist
    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import int8_mixed_precision_03_b300 as i8

    w = synth.WORKLOADS[args.workload]
    if world > 1:  # independent batches per rank
        w = w.with_(seed=w.seed + rank)
    Xh, Wh, bh = synth.make_x(w), synth.make_w(w), synth.make_bias(w)
    X = torch.from_numpy(Xh).to(device)
    bias = torch.from_numpy(bh).to(device)
    Wd = torch.from_numpy(Wh).to(device)
    CB, SCB = i8.int8_quantize_weight(Wd)        # once per weight, off the timed path
    ws = i8.alloc_workspace(w.T, w.d_in, w.d_out, device)
    Y = torch.empty((w.T, w.d_out), dtype=torch.float16, device=device)
    flush = L2Flush(device)
    zp = args.zeropoint
    if zp:   # zeropoint activation codes; the weight's code sums are prepared with CB
        sums = i8.int8_weight_code_sums(CB)

    def matmul(x, y, wsp):
        if zp:
            i8.int8_matmul_zeropoint(x, CB, SCB, sums, w.threshold, bias, Y=y, workspace=wsp)
        else:
            i8.int8_matmul(x, CB, SCB, w.threshold, bias, Y=y, workspace=wsp)

    def step():
        matmul(X, Y, ws)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if i8.i8_get_status(ws) != 0:
        raise RuntimeError(f"device status {i8.i8_get_status(ws)} after warm-up")

    K = args.steps
    # per-step events around the whole step, plus events between the three kernels (the
    # roofline's kernel time comes from the same timed region)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for e in [x for row in ev for x in row] + ends:   # create the CUDA events before timing
        e.record()
    torch.cuda.synchronize()
    clocks = ClockSampler(local) if rank == 0 else None
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.mark_start()
    launches = 0
    for k in range(K):
        flush(k)                                  # L2 flush between timed steps (not timed)
        i8.i8_set_profile_events(ev[k])
        step()
        launches += 3                             # our kernels: colstats, quantize, matmul
        ends[k].record()
    i8.i8_set_profile_events(None)
    torch.cuda.synchronize()
    if clocks:
        clocks.mark_end()
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    if i8.i8_get_status(ws) != 0:
        raise RuntimeError(f"device status {i8.i8_get_status(ws)} in the timed region")
    step_ms = [ev[k][0].elapsed_time(ends[k]) for k in range(K)]
    k_ms = {"colstats": [ev[k][0].elapsed_time(ev[k][1]) for k in range(K)],
            "quantize_gather": [ev[k][1].elapsed_time(ev[k][2]) for k in range(K)],
            "matmul": [ev[k][2].elapsed_time(ev[k][3]) for k in range(K)]}
    local_s = sum(step_ms) / 1e3
    ops = workload_ops(w)
    total_s, total_ops = aggregate(local_s, ops * K)
    value = total_ops / total_s / 1e12

    # End to end through the public API: every step copies its X in from pinned host memory
    # and its Y back to pinned host memory. Steps alternate between two streams with their
    # own device buffers, so one step's input copy overlaps the previous step's matmul and
    # output copy (the copy engines of the two directions run concurrently).
    Xpin = torch.from_numpy(Xh).pin_memory()
    nbuf = 2
    streams = [torch.cuda.Stream(device) for _ in range(nbuf)]
    Xe = [torch.empty_like(X) for _ in range(nbuf)]
    Ye = [torch.empty((w.T, w.d_out), dtype=torch.float16, device=device) for _ in range(nbuf)]
    Ype = [torch.empty((w.T, w.d_out), dtype=torch.float16).pin_memory() for _ in range(nbuf)]
    wse = [ws] + [i8.alloc_workspace(w.T, w.d_in, w.d_out, device) for _ in range(nbuf - 1)]
    Ke = min(K, 50)

    def e2e_steps(n):
        start = torch.cuda.current_stream(device)
        for st in streams:
            st.wait_stream(start)
        for k in range(n):
            b = k % nbuf
            with torch.cuda.stream(streams[b]):
                Xe[b].copy_(Xpin, non_blocking=True)
                matmul(Xe[b], Ye[b], wse[b])
                Ype[b].copy_(Ye[b], non_blocking=True)
        for st in streams:
            start.wait_stream(st)

    e2e_steps(2 * nbuf)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    e2e_steps(Ke)
    e1.record()
    torch.cuda.synchronize()
    for b in range(nbuf):
        if i8.i8_get_status(wse[b]) != 0:
            raise RuntimeError(f"device status {i8.i8_get_status(wse[b])} in the e2e run")
    e2e_s, e2e_ops = aggregate(e0.elapsed_time(e1) / 1e3, ops * Ke)
    Ypin = Ype[0]

    # our fp16 GEMM on the same shape (the 16-bit comparator), L2 flushed between launches
    f16_ms = event_time_us(lambda: i8.f16_matmul(X, Wd, bias, Y=Y), flush, Ke) / 1e3
    del Wd
    # Streaming references at the same sizes, timed the same way: reading X (the column
    # statistics read X once) and an fp16 -> fp16 copy of X (the quantize pass reads X and
    # writes codes of the same size); what any single launch of that traffic takes here.
    Xc = torch.empty(X.shape, dtype=torch.int8 if uses_gemv(w) else torch.float16,
                     device=device)
    ref_us = {"colstats": event_time_us(lambda: torch.amax(X), flush, Ke),
              "quantize_gather": event_time_us(lambda: Xc.copy_(X), flush, Ke)}
    del Xc

    if rank != 0:
        dist.destroy_process_group()
        return
    peaks, peak_src = load_peaks()
    roof = roofline(w, statistics.mean(k_ms["matmul"]), peaks, peak_src, zp)
    line = {
        "metric": METRIC.replace("int8_matmul", "int8_matmul_zeropoint") if zp else METRIC,
        "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_s / K * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "s8", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "d_in": w.d_in, "d_out": w.d_out,
                   "threshold": w.threshold, "n_outlier_cols": w.n_outlier_cols,
                   "activation_codes": "zeropoint" if zp else "absmax",
                   "parallelism": f"replicas{world}" if world > 1 else "single",
                   "l2": L2_NOTE},
        "kernels_us": {k: round(statistics.mean(v) * 1e3, 2) for k, v in k_ms.items()},
        "prepass_gbs": prepass_gbs(w, k_ms, ref_us, peaks),
        "roofline": roof,
        "e2e": {"value": e2e_ops / e2e_s / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": int(Xpin.numel() * 2),
                "d2h_bytes_per_step": int(Ypin.numel() * 2),
                "steps": Ke, "overlap": "2 streams: a step's copies overlap its neighbours"},
        "f16_comparator": {"us": round(f16_ms * 1e3, 2),
                           "TFLOP/s": ops / (f16_ms / 1e3) / 1e12,
                           "frac_of_bf16_peak": ops / (f16_ms / 1e3) / 1e12
                           / float(peaks["bf16_tflops"]),
                           "int8_step_speedup": f16_ms / (total_s / K * 1e3)},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        CBo, SCBo = oracle.quantize_weight(Wh)
        line["cpu_baseline"] = cpu_baseline_sample(w, Xh, CBo, SCBo, bh, os.cpu_count() or 1,
                                                   zeropoint=zp)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_ffn(args) -> None:
    """The FFN block (int8_ffn) on one GPU: up projection with ReLU and the down
    projection's column flags in its epilogue, mask compaction, down projection."""
    import torch
    import int8_mixed_precision_03_b300 as i8
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    f = synth.FFN_WORKLOADS[args.ffn_workload]
    blk = synth.make_ffn(f)
    X = torch.from_numpy(blk["X"]).to(device)
    bu, bd = (torch.from_numpy(blk[k]).to(device) for k in ("b_up", "b_down"))
    Wu, Wd = (torch.from_numpy(blk[k]).to(device) for k in ("W_up", "W_down"))
    CBu, SCBu = i8.int8_quantize_weight(Wu)
    CBd, SCBd = i8.int8_quantize_weight(Wd)
    ws = torch.empty(i8.int8_ffn_workspace_size(f.T, f.d_model, f.d_ff), dtype=torch.uint8,
                     device=device)
    H = torch.empty((f.T, f.d_ff), dtype=torch.float16, device=device)
    Y = torch.empty((f.T, f.d_model), dtype=torch.float16, device=device)
    flush = L2Flush(device)
    thr = f.threshold

    def step(x=X, h=H, y=Y, w=ws):
        i8.int8_ffn(x, CBu, SCBu, CBd, SCBd, thr, bu, bd, "relu", H=h, Y=y, workspace=w)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if i8.i8_get_status(ws) != 0:
        raise RuntimeError(f"device status {i8.i8_get_status(ws)} after warm-up")
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(K)]
    st = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    en = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for e in [x for row in ev for x in row] + st + en:
        e.record()
    torch.cuda.synchronize()
    clocks = ClockSampler(0)
    torch.cuda.synchronize()
    clocks.mark_start()
    launches = 0
    for k in range(K):
        flush(k)                                  # L2 flush between timed steps (not timed)
        i8.i8_set_profile_events(ev[k])
        st[k].record()
        step()
        en[k].record()
        launches += 6    # statistics, quantize, matmul of the up projection; mask
                         # compaction, quantize, matmul of the down projection
    i8.i8_set_profile_events(None)
    torch.cuda.synchronize()
    clocks.mark_end()
    clk = clocks.stop()
    if i8.i8_get_status(ws) != 0:
        raise RuntimeError(f"device status {i8.i8_get_status(ws)} in the timed region")
    step_ms = statistics.mean(st[k].elapsed_time(en[k]) for k in range(K))
    names = ["up_colstats", "up_quantize_gather", "up_matmul", "down_mask_index",
             "down_quantize_gather", "down_matmul"]
    pairs = [(0, 1), (1, 2), (2, 3), (4, 5), (5, 6), (6, 7)]
    k_ms = {n: statistics.mean(ev[k][a].elapsed_time(ev[k][b]) for k in range(K))
            for n, (a, b) in zip(names, pairs)}
    ops = 4.0 * f.T * f.d_model * f.d_ff
    value = ops / (step_ms / 1e3) / 1e12

    def timed(fn, n):
        return event_time_us(fn, flush, n) / 1e3

    Kc = min(K, 50)
    ws_u = i8.alloc_workspace(f.T, f.d_model, f.d_ff, device)
    ws_d = i8.alloc_workspace(f.T, f.d_ff, f.d_model, device)
    H2, Y2 = torch.empty_like(H), torch.empty_like(Y)

    def two_calls():  # the same block without the fused statistics (torch ReLU between)
        i8.int8_matmul(X, CBu, SCBu, thr, bu, Y=H2, workspace=ws_u)
        torch.relu_(H2)
        i8.int8_matmul(H2, CBd, SCBd, thr, bd, Y=Y2, workspace=ws_d)

    two_ms = timed(two_calls, Kc)
    f16_ms = timed(lambda: i8.f16_ffn(X, Wu, Wd, bu, bd, "relu", H=H2, Y=Y2), Kc)

    # end to end through the public call: X in from pinned host memory, Y back, two streams
    Xpin = torch.from_numpy(blk["X"]).pin_memory()
    nbuf = 2
    streams = [torch.cuda.Stream(device) for _ in range(nbuf)]
    Xe = [torch.empty_like(X) for _ in range(nbuf)]
    He = [torch.empty_like(H) for _ in range(nbuf)]
    Ye = [torch.empty_like(Y) for _ in range(nbuf)]
    Ype = [torch.empty(Y.shape, dtype=torch.float16).pin_memory() for _ in range(nbuf)]
    wse = [ws] + [torch.empty_like(ws) for _ in range(nbuf - 1)]

    def e2e_steps(n):
        start = torch.cuda.current_stream(device)
        for s_ in streams:
            s_.wait_stream(start)
        for k in range(n):
            b = k % nbuf
            with torch.cuda.stream(streams[b]):
                Xe[b].copy_(Xpin, non_blocking=True)
                step(Xe[b], He[b], Ye[b], wse[b])
                Ype[b].copy_(Ye[b], non_blocking=True)
        for s_ in streams:
            start.wait_stream(s_)

    e2e_steps(2 * nbuf)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    e2e_steps(Kc)
    e1.record()
    torch.cuda.synchronize()
    for b in range(nbuf):
        if i8.i8_get_status(wse[b]) != 0:
            raise RuntimeError(f"device status {i8.i8_get_status(wse[b])} in the e2e run")
    e2e_s = e0.elapsed_time(e1) / 1e3

    peaks, peak_src = load_peaks()
    mm_ms = k_ms["up_matmul"] + k_ms["down_matmul"]
    achieved = ops / (mm_ms / 1e3) / 1e12
    peak = float(peaks["bf16_tflops"])
    line = {
        "metric": FFN_METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": K,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "s8", "data": "synthetic",
        "config": {"workload": f.name, "T": f.T, "d_model": f.d_model, "d_ff": f.d_ff,
                   "threshold": thr, "act": "relu",
                   "n_outlier_cols_x": f.x_workload().n_outlier_cols,
                   "n_outlier_features_h": f.n_h_outliers(), "parallelism": "single",
                   "l2": L2_NOTE},
        "kernels_us": {k: round(v * 1e3, 2) for k, v in k_ms.items()},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "traffic": None,
                     "kernel": "i8_gemm_kernel (both projections; the up projection's "
                               "epilogue with ReLU and the down projection's column flags)",
                     "peak_source": f"bf16_tflops burst, {peak_src} (MEASURED_PEAKS.json)"},
        "two_call_us": round(two_ms * 1e3, 2),
        "fusion_speedup": two_ms / step_ms,
        "f16_comparator": {"us": round(f16_ms * 1e3, 2),
                           "TFLOP/s": ops / (f16_ms / 1e3) / 1e12,
                           "frac_of_bf16_peak": ops / (f16_ms / 1e3) / 1e12 / peak,
                           "int8_step_speedup": f16_ms / step_ms},
        "e2e": {"value": ops * Kc / e2e_s / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": int(Xpin.numel() * 2),
                "d2h_bytes_per_step": int(Ype[0].numel() * 2), "steps": Kc,
                "overlap": "2 streams: a step's copies overlap its neighbours"},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = ffn_cpu_baseline(f, blk, os.cpu_count() or 1)
    print(json.dumps(line), flush=True)


def run_rows(args) -> None:
    """Standalone quantizers, HBM-bound, reported in GB/s: row-wise absmax and zeropoint and
    block-wise absmax (blocks of 64 and 128) on the sweep's X [1024, 8192] (absmax on N(0,1)
    with the sweep's outliers, zeropoint on |N(0,1)|), and the same on 16 times as many rows
    (268 MB of input, twice the L2), where one launch's fixed cost no longer dominates.
    Beside each, the time of a plain fp16 -> int8 copy of X timed the same way: the same
    traffic (2 bytes read and 1 written per value) through a library streaming kernel."""
    import torch
    import int8_mixed_precision_03_b300 as i8
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    peaks, peak_src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    flush = L2Flush(device)
    base = synth.WORKLOADS["sweep_f0.1_thr6"]
    for rows in (base.T, 16 * base.T):
        w = base.with_(T=rows)
        Xa = torch.from_numpy(synth.make_x(w)).to(device)
        Xz = torch.from_numpy(synth.make_relu_like(w)).to(device)
        cols = w.d_in
        Qc = torch.empty((rows, cols), dtype=torch.int8, device=device)
        ref_us = event_time_us(lambda: Qc.copy_(Xa), flush, args.steps, max(args.warmup, 3))
        cases = [("absmax_quantize_rows", lambda: i8.absmax_quantize_rows(Xa), 4 * rows),
                 ("zeropoint_quantize_rows", lambda: i8.zeropoint_quantize_rows(Xz), 8 * rows),
                 ("absmax_quantize_blocks[64]", lambda: i8.absmax_quantize_blocks(Xa, 64),
                  4 * rows * cols // 64),
                 ("absmax_quantize_blocks[128]", lambda: i8.absmax_quantize_blocks(Xa, 128),
                  4 * rows * cols // 128)]
        for name, fn, scale_bytes in cases:
            us = event_time_us(fn, flush, args.steps, max(args.warmup, 3))
            nbytes = 2 * rows * cols + rows * cols + scale_bytes
            gbs = nbytes / (us / 1e6) / 1e9
            print(json.dumps({
                "metric": f"{name} GB/s", "value": gbs, "unit": "GB/s", "n_gpus": 1,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3,
                "higher_is_better": True, "dtype": "s8", "data": "synthetic",
                "config": {"workload": f"{name} [{rows}, {cols}]", "l2": L2_NOTE},
                "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                             "frac": gbs / hbm, "traffic": None, "algorithmic_bytes": nbytes,
                             "peak_source": f"hbm_gbs, {peak_src} (MEASURED_PEAKS.json)"},
                "streaming_reference": {"kernel": "torch fp16 -> int8 copy of X",
                                        "us": round(ref_us, 2),
                                        "frac_of_hbm": 3 * rows * cols / (ref_us / 1e6) / 1e9 / hbm,
                                        "ours_vs_reference": ref_us / us}}), flush=True)
        del Xa, Xz, Qc
        torch.cuda.empty_cache()


def prepass_gbs(w, k_ms: dict, ref_us: dict, peaks: dict) -> dict:
    """Bandwidth of the two passes before the matmul: the column statistics read X
    (2 T in bytes); the quantize pass reads X and writes the codes (fp16 for the tensor-core
    matmul, int8 for the decode kernels) and the row scales. Beside each, the time of a
    library streaming kernel with the same traffic timed the same way (ref_us)."""
    hbm = float(peaks["hbm_gbs"])
    code_bytes = 1 if uses_gemv(w) else 2
    nb = {"colstats": 2 * w.T * w.d_in,
          "quantize_gather": 2 * w.T * w.d_in + code_bytes * w.T * w.d_in + 4 * w.T}
    out = {}
    for k, b in nb.items():
        us = statistics.mean(k_ms[k]) * 1e3
        out[k] = {"us": round(us, 2), "algorithmic_bytes": b, "gbs": b / (us / 1e6) / 1e9,
                  "frac_of_hbm": b / (us / 1e6) / 1e9 / hbm,
                  "reference_us": round(ref_us[k], 2), "ours_vs_reference": ref_us[k] / us}
    return out


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--ref-budget-s", type=float, default=120.0,
                    help="wall-clock budget of the reference arm's warm-up + timed steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--all", action="store_true",
                    help="one line per configuration (1 GPU, no CPU baseline)")
    ap.add_argument("--ffn", action="store_true", help="only the FFN block line (1 GPU)")
    ap.add_argument("--rows", action="store_true",
                    help="only the standalone quantizer lines (1 GPU)")
    ap.add_argument("--zeropoint", action="store_true",
                    help="zeropoint activation codes (int8_matmul_zeropoint)")
    ap.add_argument("--ffn-workload", default=DEFAULT_FFN, choices=sorted(synth.FFN_WORKLOADS))
    args = ap.parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    elif args.all:
        if dist_env()[1] > 1:
            raise SystemExit("--all runs on one GPU")
        args.no_cpu_baseline = True
        for name in ALL_CONFIGS:
            args.workload = name
            run_ours(args)
        args.workload, args.zeropoint = DEFAULT_WORKLOAD, True
        run_ours(args)
        args.zeropoint = False
        run_ffn(args)
        run_rows(args)
    elif args.rows:
        run_rows(args)
    elif args.ffn:
        if dist_env()[1] > 1:
            raise SystemExit("--ffn runs on one GPU")
        run_ffn(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
