"""SGEMM benchmark: GFLOP/s of C = alpha * A.B + beta * C, device-timed, one JSON line.

Default workload: M = N = K = 4096 fp32 row-major, A, B, C ~ U[-1, 1) from seed 0, alpha = 1,
beta = 0 (the pages' headline problem, 137.4 GFLOP per call). A "step" is one library call.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload headline|sq256|edge0..edge3|sweepNNNN|llm_qkv|llm_up|llm_down|llm_head]
                  [--path simt|3xtf32|tf32]

Timing: W untimed warm-up steps, then K steps. Before every step a 256 MiB buffer is written
(L2 is 129 MB) so each step starts with cold L2; each step's GEMM is bracketed by CUDA
events on the stream it runs on. value = 2*M*N*K * K_steps * ranks / max over ranks of the
summed GEMM time. Under torchrun (N > 1) every rank runs its own replica of the workload
(the method shards without communication; no collective is on the data path) and the max
of the per-rank times is taken through the process group.

The reference arm (--impl reference) times the CPU oracle (fp64 triple loop, all host cores)
on a bounded row sample of the same workload, each step one sample.
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
from pathlib import Path

ROOT = Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

METRIC = "SGEMM GFLOP/s at 4096³ fp32 and % of GB300 FP32 peak (1 GPU, device-timed)"
UNIT = "GFLOP/s"
BOOST_MHZ = 2070.0          # GB300 maximum SM clock (the SIMT peak's clock)
FMA_PER_CLK_PER_SM = 128    # FP32 lanes per SM
TF32_NOMINAL_TFLOPS = 1100.0  # nominal dense TF32 tensor rate of a GB300
BF16_NOMINAL_TFLOPS = 2250.0  # nominal dense BF16 rate (the ratio scales the measured bf16 peak)
L2_FLUSH_BYTES = 256 << 20

WORKLOADS = {
    "headline": dict(M=4096, N=4096, K=4096, alpha=1.0, beta=0.0, dist="uniform"),
    "sq256": dict(M=256, N=256, K=256, alpha=1.0, beta=0.0, dist="uniform"),
    "sq256_ab": dict(M=256, N=256, K=256, alpha=1.5, beta=-0.5, dist="uniform"),
    "edge0": dict(M=4095, N=3001, K=1537, alpha=0.7, beta=-1.3, dist="normal"),
    "edge1": dict(M=1, N=4096, K=4096, alpha=0.7, beta=-1.3, dist="normal"),
    "edge2": dict(M=4096, N=1, K=4096, alpha=0.7, beta=-1.3, dist="normal"),
    "edge3": dict(M=127, N=129, K=4099, alpha=0.7, beta=-1.3, dist="normal"),
    "llm_qkv": dict(M=16384, N=12288, K=4096, alpha=1.0, beta=1.0, dist="llm"),
    "llm_up": dict(M=16384, N=14336, K=4096, alpha=1.0, beta=1.0, dist="llm"),
    "llm_down": dict(M=16384, N=4096, K=14336, alpha=1.0, beta=1.0, dist="llm"),
    "llm_head": dict(M=16384, N=32000, K=4096, alpha=1.0, beta=1.0, dist="llm"),
}
for _n in (128, 256, 512, 1024, 2048, 4096, 8192, 16384):
    WORKLOADS[f"sweep{_n}"] = dict(M=_n, N=_n, K=_n, alpha=1.0, beta=0.0, dist="uniform")


def host_inputs(w, seed=0):
    import synth
    M, N, K = w["M"], w["N"], w["K"]
    if w["dist"] == "uniform":
        return synth.uniform(M, K, seed), synth.uniform(K, N, seed + 1), synth.uniform(M, N, seed + 2)
    if w["dist"] == "normal":
        return synth.normal(M, K, seed), synth.normal(K, N, seed + 1), synth.normal(M, N, seed + 2)
    if w["dist"] == "llm":
        return (synth.normal(M, K, seed), synth.normal(K, N, seed + 1, sigma=0.02),
                synth.normal(M, N, seed + 2))
    raise ValueError(w["dist"])


def workload_name(name, w):
    return f"sgemm_{name}_{w['M']}x{w['N']}x{w['K']}_alpha{w['alpha']:g}_beta{w['beta']:g}"


# ---- distributed plumbing (replicas) ----------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_group(world, backend):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(value: float, dist, device=None) -> float:
    """Maximum of a per-rank float across the process group (identity without one)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---- clocks --------------------------------------------------------------------------------------

_REASON_BITS = {
    0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
    0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
    0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting",
}


class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons while the timed region runs."""

    def __init__(self, index: int, period_ms: int = 100):
        self.index, self.period_ms = index, period_ms
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (FileNotFoundError, OSError):
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
            self._t.join(timeout=2)

    def summary(self):
        mhz, maxes, reasons = [], [], set()
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 4:
                continue
            try:
                mhz.append(float(parts[0]))
                maxes.append(float(parts[1]))
                bits = int(parts[3], 16) if parts[3].startswith("0x") else int(parts[3])
            except ValueError:
                continue
            for bit, name in _REASON_BITS.items():
                if bits & bit:
                    reasons.add(name)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max(maxes),
                "reasons": sorted(reasons), "samples": len(mhz)}


# ---- profiles (ncu traffic figures committed under profiles/) --------------------------------------

KERNEL_SOURCES = {
    "simt": ("simt_gemm.cu", "simt_gemm.cuh", "ptx.cuh"),
    "3xtf32": ("tf32x3_gemm.cu", "tf32x3_gemm.cuh", "ptx.cuh"),
}


def source_hash(path: str = "simt") -> str:
    """Hash of the source files that define a path's kernels (ncu figures go stale with them)."""
    h = hashlib.sha256()
    csrc = ROOT / "dense_fp32_gemm_08_gb300" / "csrc"
    for name in KERNEL_SOURCES[path]:
        p = csrc / name
        if p.exists():
            h.update(name.encode())
            h.update(p.read_bytes())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str, path: str = "simt"):
    """DRAM bytes per launch from profiles/ncu_traffic.json, or None when absent or taken on
    a different kernel source."""
    fname = ROOT / "profiles" / "ncu_traffic.json"
    if not fname.exists():
        return None
    try:
        data = json.loads(fname.read_text())
    except json.JSONDecodeError:
        return None
    entry = data.get(f"{kernel}@{workload}")
    if not entry or entry.get("source_hash") != source_hash(path):
        return None
    return entry.get("dram_bytes_per_launch")


def measured_peaks():
    path = ROOT / "MEASURED_PEAKS.json"
    if path.exists():
        try:
            return json.loads(path.read_text())
        except json.JSONDecodeError:
            return {}
    return {}


# ---- CPU oracle baseline -------------------------------------------------------------------------

class OracleTimer:
    """Times the CPU oracle on seeded row samples of a workload (all N columns, full K)."""

    def __init__(self, w, A, B, C):
        import numpy as np
        import oracle
        self.w, self.A, self.B, self.C = w, A, B, C
        self.oracle = oracle
        self.threads = oracle.max_threads()
        self.rng = np.random.default_rng(0)
        self.np = np
        self.per_row = None

    def run(self, nrows: int) -> tuple[float, int]:
        w = self.w
        M, N, K = w["M"], w["N"], w["K"]
        rows = self.np.sort(self.rng.choice(M, size=min(nrows, M), replace=False))
        beta = w["beta"]
        t0 = time.perf_counter()
        self.oracle.sgemm(M, N, K, w["alpha"], self.A, K, self.B, N, beta,
                          self.C if beta != 0.0 else None, N, rows=rows)
        return time.perf_counter() - t0, len(rows)

    def rows_for(self, seconds: float) -> int:
        if self.per_row is None:
            probe = max(1, min(self.w["M"], self.threads))
            dt, n = self.run(probe)
            self.per_row = max(dt / n, 1e-7)
        return int(min(self.w["M"], max(1, seconds / self.per_row)))


def oracle_sample(w, target_s: float, A, B, C, threads: int | None = None):
    """Times the oracle on a row sample sized for about `target_s` seconds, on `threads`
    OpenMP threads (default: all). Returns (gflops, seconds, rows, threads)."""
    import oracle
    full = oracle.max_threads()
    if threads is not None:
        oracle.set_threads(threads)
    try:
        t = OracleTimer(w, A, B, C)
        if threads is not None:
            t.threads = threads
        dt, n = t.run(t.rows_for(target_s))
    finally:
        oracle.set_threads(full)
    return 2.0 * n * w["N"] * w["K"] / dt / 1e9, dt, n, t.threads


# ---- our arm ---------------------------------------------------------------------------------------

def run_ours(args):
    import torch
    import dense_fp32_gemm_08_gb300 as sg

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = init_group(world, "nccl")
    dev = torch.device("cuda", local)
    w = WORKLOADS[args.workload]
    M, N, K, alpha, beta = w["M"], w["N"], w["K"], w["alpha"], w["beta"]
    flops = 2.0 * M * N * K
    entry = {"simt": sg.sgemm, "3xtf32": sg.sgemm_3xtf32, "tf32": sg.sgemm_tf32}[args.path]

    A_h, B_h, C_h = host_inputs(w)
    A = torch.from_numpy(A_h).to(dev)
    B = torch.from_numpy(B_h).to(dev)
    C = torch.from_numpy(C_h).to(dev)
    C0 = C.clone() if beta != 0.0 else None
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    cfg_id = sg.sgemm_select_config(M, N, K, alpha, A, K, B, N, C, N)
    kernel = (sg.sgemm_config_name(cfg_id) if args.path == "simt"
              else {"3xtf32": "tf32x3_tcgen05", "tf32": "tf32_tcgen05"}[args.path])

    def step():
        entry(M, N, K, alpha, A, K, B, N, beta, C, N, stream)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        if C0 is not None:
            C.copy_(C0)
        step()
    torch.cuda.synchronize(dev)
    if sg.sgemm_device_status(stream) != sg.SGEMM_OK:
        raise RuntimeError(f"device status after warm-up: {sg.sgemm_last_error()}")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(dist)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clocks:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(float(i))
            if C0 is not None:   # beta != 0: restore C so every step computes the same thing
                C.copy_(C0)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - wall0
    barrier(dist)
    if sg.sgemm_device_status(stream) != sg.SGEMM_OK:
        raise RuntimeError(f"device status after timing: {sg.sgemm_last_error()}")
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = max_over_ranks(sum(step_ms), dist, dev)
    value = flops * args.steps * world / (total_ms / 1e3) / 1e9

    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    clk = clocks.summary()
    peak_boost = sms * BOOST_MHZ * 1e6 * FMA_PER_CLK_PER_SM * 2 / 1e12   # TFLOP/s
    avg_ms = sum(step_ms) / len(step_ms)
    achieved_tflops = flops / (avg_ms / 1e3) / 1e12
    if args.path == "simt":
        roof = {"bound": "alu", "achieved": round(achieved_tflops, 3), "peak": round(peak_boost, 3),
                "unit": "TFLOP/s", "frac": round(achieved_tflops / peak_boost, 4),
                "traffic": ncu_traffic(kernel, args.workload, "simt"),
                "peak_basis": f"{sms} SMs x {BOOST_MHZ:.0f} MHz x {FMA_PER_CLK_PER_SM} FMA/clk x 2"}
        if clk.get("sm_mhz"):
            roof["frac_at_run_clock"] = round(
                achieved_tflops / (sms * clk["sm_mhz"] * 1e6 * FMA_PER_CLK_PER_SM * 2 / 1e12), 4)
    else:
        products = 3 if args.path == "3xtf32" else 1
        peaks = measured_peaks()
        if peaks.get("bf16_tflops"):
            tf32_peak = peaks["bf16_tflops"] * TF32_NOMINAL_TFLOPS / BF16_NOMINAL_TFLOPS
            basis = (f"measured bf16 {peaks['bf16_tflops']} TFLOP/s x nominal TF32:BF16 "
                     f"{TF32_NOMINAL_TFLOPS:g}:{BF16_NOMINAL_TFLOPS:g}")
        else:
            tf32_peak = TF32_NOMINAL_TFLOPS
            basis = "nominal dense TF32 rate (no measured peak file)"
        roof = {"bound": "tensor", "achieved": round(achieved_tflops, 3),
                "peak": round(tf32_peak, 1), "unit": "TFLOP/s",
                "frac": round(achieved_tflops / tf32_peak, 4),
                "issued_tflops": round(products * achieved_tflops, 3),
                "issued_frac": round(products * achieved_tflops / tf32_peak, 4),
                "traffic": ncu_traffic(kernel, args.workload, "3xtf32"),
                "peak_basis": basis + f"; achieved counts 2MNK, issued counts the {products} "
                                      "TF32 product(s) per multiply-add",
                "frac_of_fp32_simt_peak": round(achieved_tflops / peak_boost, 4)}

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, torch, sg, dev, stream, w, A_h, B_h, C_h, entry, dist, world)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_name(args.workload, w), "M": M, "N": N, "K": K,
                   "alpha": alpha, "beta": beta, "inputs": w["dist"] + ", seed 0",
                   "path": args.path, "kernel": kernel,
                   "l2": "flushed before every step (256 MiB write)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "gflops_median": round(flops / (statistics.median(step_ms) / 1e3) / 1e9, 1),
        "gflops_best": round(flops / (min(step_ms) / 1e3) / 1e9, 1),
        "pct_fp32_simt_peak_boost": round(100.0 * value / world / (peak_boost * 1e3), 2),
        "roofline": roof,
        "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
        "clock_samples": clk["samples"],
        "gpu_launches": args.steps * launches_per_call(args.path, kernel, w),
        "wall_s_timed_loop": round(wall, 4),
        "e2e": e2e,
        "device": props.name, "sms": sms,
    }
    if rank == 0 and not args.no_cublas_context:
        line["context_cublas"] = cublas_context(torch, dev, stream, w, A, B, C, C0, flush,
                                                max(3, args.warmup), min(args.steps, 50),
                                                value / world)
    if rank == 0 and not args.no_cpu_baseline:
        gf, dt, nrows, threads = oracle_sample(w, args.cpu_seconds, A_h, B_h, C_h)
        line["cpu_baseline"] = {"value": round(gf, 3), "unit": UNIT, "cores": threads,
                                "kind": "oracle",
                                "sample": f"{nrows} of {M} result rows (all N columns, full K), "
                                          f"{dt:.1f} s, fp64 triple loop, OpenMP over rows"}
        gf1, dt1, n1, _ = oracle_sample(w, args.cpu_seconds / 4, A_h, B_h, C_h, threads=1)
        line["cpu_baseline"]["single_core"] = {
            "value": round(gf1, 3), "unit": UNIT, "cores": 1,
            "sample": f"{n1} of {M} result rows (all N columns, full K), {dt1:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def launches_per_call(path: str, kernel: str, w) -> int:
    """Kernels one library call launches for the bench's operands (lda = K, ldb = N,
    ldc = N, 16-byte-aligned allocations): the tensor paths split A, split-and-transpose B,
    then run the GEMM; a repacked SIMT configuration first copies each operand whose rows
    TMA cannot read (K or N not a multiple of 4) into aligned storage."""
    if path in ("3xtf32", "tf32"):
        return 3
    n = 1
    if kernel.startswith("packed"):
        n += int(w["K"] % 4 != 0) + int(w["N"] % 4 != 0)
    return n


def cublas_context(torch, dev, stream, w, A, B, C, C0, flush, warmup, steps, ours):
    """The same workload through torch.addmm (cuBLAS SGEMM, TF32 off) under the same timing
    rules: a comparison bar only, never a path of the library."""
    M, N, K, alpha, beta = w["M"], w["N"], w["K"], w["alpha"], w["beta"]
    flops = 2.0 * M * N * K
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    out = torch.empty_like(C)
    src = C0 if C0 is not None else C
    try:
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                flush.fill_(1.0)
                torch.addmm(src, A, B, beta=beta, alpha=alpha, out=out)
            ms = []
            for i in range(steps):
                flush.fill_(float(i))
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                torch.addmm(src, A, B, beta=beta, alpha=alpha, out=out)
                e1.record(stream)
                e1.synchronize()
                ms.append(e0.elapsed_time(e1))
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    gf = flops * len(ms) / (sum(ms) / 1e3) / 1e9
    return {"value": round(gf, 1), "unit": UNIT, "library": "torch.addmm (cuBLAS SGEMM), TF32 off",
            "steps": len(ms), "ours_over_it": round(ours / gf, 3)}


def run_e2e(args, torch, sg, dev, stream, w, A_h, B_h, C_h, entry, dist, world):
    """Same metric through the public host-memory entry point: each step is one sgemm_host
    call on pinned host buffers, which uploads A and B (and C when beta != 0), computes, and
    returns when C is back in host memory (chunked so copies overlap the device work).
    Timed on the host clock around whole calls; the tensor paths copy and call in turn."""
    M, N, K, alpha, beta = w["M"], w["N"], w["K"], w["alpha"], w["beta"]
    flops = 2.0 * M * N * K
    A_p = torch.from_numpy(A_h).pin_memory()
    B_p = torch.from_numpy(B_h).pin_memory()
    C_p = torch.from_numpy(C_h).pin_memory()
    h2d = (M * K + K * N + (M * N if beta != 0.0 else 0)) * 4
    d2h = M * N * 4
    if args.path == "simt":
        def step():
            sg.sgemm_host(M, N, K, alpha, A_p, K, B_p, N, beta, C_p, N, stream)
        how = "sgemm_host on pinned buffers (chunked, copies overlap compute)"
    else:
        A = torch.empty((M, K), dtype=torch.float32, device=dev)
        B = torch.empty((K, N), dtype=torch.float32, device=dev)
        C = torch.empty((M, N), dtype=torch.float32, device=dev)

        def step():
            A.copy_(A_p, non_blocking=True)
            B.copy_(B_p, non_blocking=True)
            if beta != 0.0:
                C.copy_(C_p, non_blocking=True)
            entry(M, N, K, alpha, A, K, B, N, beta, C, N, stream)
            C_p.copy_(C, non_blocking=True)
            torch.cuda.synchronize(dev)
        how = "copies to device, device call, copy back (pinned buffers)"

    for _ in range(max(2, args.warmup // 2)):
        step()
    torch.cuda.synchronize(dev)
    n = max(3, min(args.steps, args.e2e_steps))
    barrier(dist)
    t0 = time.perf_counter()
    for _ in range(n):
        step()
    torch.cuda.synchronize(dev)
    ms = max_over_ranks((time.perf_counter() - t0) * 1e3, dist, dev)
    if sg.sgemm_device_status(stream) != sg.SGEMM_OK:
        raise RuntimeError("device status after e2e timing")
    return {"value": round(flops * n * world / (ms / 1e3) / 1e9, 1), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "ms_per_step": round(ms / n, 4), "host_buffers": "pinned", "how": how}


# ---- reference arm: the CPU oracle -----------------------------------------------------------------

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    M, N, K = w["M"], w["N"], w["K"]
    A_h, B_h, C_h = host_inputs(w)
    timer = OracleTimer(w, A_h, B_h, C_h)
    # the whole run (warm-up + steps) stays near `cpu_seconds` of oracle work, >= 1 row a step
    per_step = min(5.0, max(0.02, args.cpu_seconds / (args.steps + args.warmup)))
    nrows = timer.rows_for(per_step)
    for _ in range(args.warmup):
        timer.run(nrows)
    total_flop, total_s = 0.0, 0.0
    for _ in range(args.steps):
        dt, n = timer.run(nrows)
        total_flop += 2.0 * n * N * K
        total_s += dt
    threads = timer.threads
    rows_seen = [nrows]
    value = total_flop / total_s / 1e9
    sample = (f"each step {min(rows_seen)}-{max(rows_seen)} of {M} result rows "
              f"(all N columns, full K), fp64 triple loop, OpenMP over rows")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total_s / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(args.workload, w), "M": M, "N": N, "K": K,
                   "alpha": w["alpha"], "beta": w["beta"], "inputs": w["dist"] + ", seed 0",
                   "path": "cpu oracle", "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def parse(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="headline")
    ap.add_argument("--path", choices=["simt", "3xtf32", "tf32"], default="simt")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cublas-context", action="store_true",
                    help="skip timing torch.addmm (cuBLAS) on the same workload")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="oracle seconds for the cpu_baseline sample (reference arm: whole run)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps < 1:
        ap.error("--steps must be >= 1")
    return args


def main(argv=None):
    args = parse(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
