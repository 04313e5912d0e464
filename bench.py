"""SGEMM benchmark: GFLOP/s of C = alpha * A.B + beta * C, device-timed, one JSON line.

Default workload: M = N = K = 4096 fp32 row-major, A, B, C ~ U[-1, 1) from seed 0, alpha = 1,
beta = 0 (the pages' headline problem, 137.4 GFLOP per call). A "step" is one library call.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload headline|sq256|edge0..edge3|sweepNNNN|llm_qkv|llm_up|llm_down|llm_head]
                  [--path simt|3xtf32|tf32] [--no-paths] [--no-sweep]

Timing: W untimed warm-up steps, then exactly K steps. Before every step a 256 MiB buffer is
written (L2 is 129 MB), so each step starts with cold L2, and another 256 MiB buffer is read,
so the lines the write left dirty are written back before the step rather than during it;
each step's GEMM is bracketed by CUDA events on the stream it runs on. A spin kernel ahead of
the steps keeps the device busy while the host queues them, so host-side delays never fall
between a start event and its launch. value = 2*M*N*K * K_steps * ranks / max over ranks of the
summed GEMM time. SM clocks and clock-event reasons are sampled in process through NVML every
2 ms during the timed steps (nvidia-smi every 20 ms as well); a `sustained` block then repeats
the step for at least one second under the same sampling. Under torchrun (N > 1) every rank
runs its own replica of the workload (the method shards without communication; no collective
is on the data path) and the max of the per-rank times is taken through the process group.

After the headline line's own measurement (and outside its timed region) the same run reports
`paths` (the 3xTF32 and TF32 tensor-core paths on the same workload, against the TF32 peak)
and `sweep` (the square sizes 128..16384, the four edge shapes and the four LLM-layer shapes
on the SIMT path, each with cuBLAS SGEMM timed beside it under the same rules; the HBM-bound
shapes also against a device copy that reads the same bytes, the copy peak's method at that
size).
Sweep inputs are drawn on the device from torch's seeded generator with the workloads'
distributions.

The CPU baseline times the oracle on a row sample of the workload; the same rows of the
timed call's result are compared with the oracle's (the `check` block) and the run fails
if they exceed the 1e-5 normalised bound.

The reference arm (--impl reference) times the CPU oracle (fp64 triple loop, all host cores)
on a bounded row sample of the same workload, each step one sample.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
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


class NvmlClocks:
    """Samples the SM clock and the clock-event reasons in process through NVML (ctypes on the
    driver's libnvidia-ml), every `period_s` seconds, while a region runs. The GPU is found by
    its UUID (falling back to the NVML index), so CUDA_VISIBLE_DEVICES renumbering is harmless.
    Reading clocks changes no setting."""

    _CLOCK_SM = 1

    def __init__(self, uuid: str | None, index: int, period_s: float = 0.002):
        self.uuid, self.index, self.period_s = uuid, index, period_s
        self.samples: list[tuple[float, int]] = []
        self.max_mhz = None
        self._lib = self._handle = self._thread = None
        self._stop = threading.Event()

    def _open(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return False
        if lib.nvmlInit_v2() != 0:
            return False
        handle = ctypes.c_void_p()
        ok = False
        if self.uuid:
            ok = lib.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(handle)) == 0
        if not ok:
            ok = lib.nvmlDeviceGetHandleByIndex_v2(self.index, ctypes.byref(handle)) == 0
        if not ok:
            return False
        self._reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(handle, self._CLOCK_SM, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        self._lib, self._handle = lib, handle
        return True

    def _run(self):
        import ctypes
        mhz, bits = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if (self._lib.nvmlDeviceGetClockInfo(self._handle, self._CLOCK_SM, ctypes.byref(mhz)) == 0
                    and self._reasons(self._handle, ctypes.byref(bits)) == 0):
                self.samples.append((float(mhz.value), int(bits.value)))
            self._stop.wait(self.period_s)

    def __enter__(self):
        try:
            if self._open():
                self._thread = threading.Thread(target=self._run, daemon=True)
                self._thread.start()
        except (OSError, AttributeError):
            self._lib = None
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._thread is not None:
            self._thread.join(timeout=2)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0}
        reasons = sorted({name for _, b in self.samples for bit, name in _REASON_BITS.items()
                          if b & bit})
        return {"sm_mhz": statistics.median(m for m, _ in self.samples),
                "sm_max_mhz": self.max_mhz or max(m for m, _ in self.samples),
                "reasons": reasons, "samples": len(self.samples)}


def merge_clocks(nvml: dict, smi: dict) -> dict:
    """The clock record of a region: NVML's in-process samples when there are any, else
    nvidia-smi's; reasons are the union of both."""
    base = nvml if nvml.get("samples") else smi
    out = {"sm_mhz": base.get("sm_mhz"), "sm_max_mhz": base.get("sm_max_mhz") or smi.get("sm_max_mhz"),
           "reasons": sorted(set(nvml.get("reasons", [])) | set(smi.get("reasons", []))),
           "samples": base.get("samples", 0), "source": "nvml" if base is nvml else "nvidia-smi",
           "smi_samples": smi.get("samples", 0)}
    return out


# ---- profiles (ncu traffic figures committed under profiles/) --------------------------------------

KERNEL_SOURCES = {
    "simt": ("simt_kernels.cuh", "simt_gemm.cu", "simt_gemm_dp.cu", "simt_gemm_dpcp.cu",
             "simt_gemm_sk.cu", "simt_gemm_sk128.cu", "simt_gemm_sk64.cu", "simt_gemm_skcp.cu",
             "simt_gemm_ck.cu", "simt_gemm.cuh", "ptx.cuh", "epilogue.cuh", "raster.cuh"),
    "3xtf32": ("tf32x3_gemm.cu", "tf32x3_gemm.cuh", "ptx.cuh", "epilogue.cuh", "raster.cuh"),
}


def code_of(text: str) -> str:
    """A C/CUDA source without its comments and with runs of whitespace collapsed: what the
    compiler sees, so that editing a comment does not mark ncu figures stale."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_hash(path: str = "simt") -> str:
    """Hash of the code of the source files that define a path's kernels (ncu figures go
    stale with it)."""
    h = hashlib.sha256()
    csrc = ROOT / "dense_fp32_gemm_08_gb300" / "csrc"
    for name in KERNEL_SOURCES[path]:
        p = csrc / name
        if p.exists():
            h.update(name.encode())
            h.update(code_of(p.read_text()).encode())
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
    """Times the CPU oracle on seeded row samples of a workload (all N columns, full K). The
    last sample's row indices and result rows are kept (`last_rows`, `last_out`)."""

    def __init__(self, w, A, B, C):
        import numpy as np
        import oracle
        self.w, self.A, self.B, self.C = w, A, B, C
        self.oracle = oracle
        self.threads = oracle.max_threads()
        self.rng = np.random.default_rng(0)
        self.np = np
        self.per_row = None
        self.last_rows = self.last_out = None

    def run(self, nrows: int) -> tuple[float, int]:
        w = self.w
        M, N, K = w["M"], w["N"], w["K"]
        rows = self.np.sort(self.rng.choice(M, size=min(nrows, M), replace=False))
        beta = w["beta"]
        t0 = time.perf_counter()
        out = self.oracle.sgemm(M, N, K, w["alpha"], self.A, K, self.B, N, beta,
                                self.C if beta != 0.0 else None, N, rows=rows)
        dt = time.perf_counter() - t0
        self.last_rows, self.last_out = rows, out
        return dt, len(rows)

    def rows_for(self, seconds: float) -> int:
        if self.per_row is None:
            probe = max(1, min(self.w["M"], self.threads))
            dt, n = self.run(probe)
            self.per_row = max(dt / n, 1e-7)
        return int(min(self.w["M"], max(1, seconds / self.per_row)))


CHECK_BOUND = 1e-5
CHECK_ROWS = 64


def result_check(w, A, B, C, rows, want, got_full):
    """Normalised error of the GPU result rows against the oracle rows just timed (at most
    CHECK_ROWS of them, spread over the sample)."""
    import numpy as np
    import oracle
    M, N, K = w["M"], w["N"], w["K"]
    pick = np.unique(np.linspace(0, len(rows) - 1, min(CHECK_ROWS, len(rows))).astype(int))
    r = rows[pick]
    den = oracle.absdot(M, N, K, A, K, B, N, rows=r)
    err = oracle.normalized_error(got_full[r], want[pick], den, w["alpha"], w["beta"],
                                  C[r] if w["beta"] != 0.0 else None)
    return {"rows": int(len(r)), "normalized_error": float(err), "bound": CHECK_BOUND,
            "ok": bool(err <= CHECK_BOUND),
            "what": "result of the timed call against the oracle rows of the cpu_baseline sample"}


def oracle_sizes(rows_cap_s: float = 0.5, sizes=(256, 1024, 2048, 8192, 16384), full_up_to=2048,
                 single_core_up_to=1024):
    """The oracle on the square sizes of the sweep, on the machine's host cores: 256^3 to 2048^3 in
    full (256^3 and 1024^3 also on one core), 8192^3 and 16384^3 on a row sample sized for
    about `rows_cap_s` seconds, extrapolated to the full size and labelled so. Inputs are drawn
    from numpy's seeded generator (uniform [-1, 1)); the oracle's time does not depend on the
    values."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(0)
    full = oracle.max_threads()
    out = []
    for n in sizes:
        A = (rng.random((n, n), dtype=np.float32) * 2 - 1)
        B = (rng.random((n, n), dtype=np.float32) * 2 - 1)
        modes = [full] + ([1] if n <= single_core_up_to else [])
        for threads in modes:
            oracle.set_threads(threads)
            try:
                if n <= full_up_to:
                    t0 = time.perf_counter()
                    oracle.sgemm(n, n, n, 1.0, A, n, B, n, 0.0, None, n)
                    dt, rows = time.perf_counter() - t0, n
                else:
                    probe = np.arange(min(n, 2 * threads))
                    t0 = time.perf_counter()
                    oracle.sgemm(n, n, n, 1.0, A, n, B, n, 0.0, None, n, rows=probe)
                    per_row = (time.perf_counter() - t0) / len(probe)
                    rows = int(min(n, max(len(probe), rows_cap_s / max(per_row, 1e-9))))
                    sample = np.sort(rng.choice(n, size=rows, replace=False))
                    t0 = time.perf_counter()
                    oracle.sgemm(n, n, n, 1.0, A, n, B, n, 0.0, None, n, rows=sample)
                    dt = time.perf_counter() - t0
            finally:
                oracle.set_threads(full)
            gf = 2.0 * rows * n * n / dt / 1e9
            out.append({"n": n, "cores": threads, "gflops": round(gf, 3),
                        "seconds_full": round(2.0 * n ** 3 / (gf * 1e9), 2),
                        "how": "full" if rows == n else
                               f"extrapolated from {rows} of {n} rows (all columns, full K)"})
        del A, B
    return out


def oracle_sample(w, target_s: float, A, B, C, threads: int | None = None, result=None):
    """Times the oracle on a row sample sized for about `target_s` seconds, on `threads`
    OpenMP threads (default: all). Returns (gflops, seconds, rows, threads, check), where
    check compares `result` (the GPU's C, when given) with the sampled oracle rows."""
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
    check = None
    if result is not None:
        check = result_check(w, A, B, C, t.last_rows, t.last_out, result)
    return 2.0 * n * w["N"] * w["K"] / dt / 1e9, dt, n, t.threads, check


def device_inputs(torch, dev, w, seed=0):
    """Sweep inputs drawn on the device from torch's seeded generator with the workload's
    distribution (uniform [-1, 1), N(0, 1), or the LLM recipe with B ~ N(0, 0.02^2))."""
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    M, N, K = w["M"], w["N"], w["K"]

    def draw(rows, cols, kind, sigma=1.0):
        if kind == "uniform":
            return torch.rand(rows, cols, generator=g, device=dev) * 2.0 - 1.0
        return torch.randn(rows, cols, generator=g, device=dev) * sigma

    if w["dist"] == "llm":
        return draw(M, K, "normal"), draw(K, N, "normal", 0.02), draw(M, N, "normal")
    return draw(M, K, w["dist"]), draw(K, N, w["dist"]), draw(M, N, w["dist"])


class L2Flush:
    """Before every timed call: write a 256 MiB buffer (evicts the call's inputs from the
    129 MB L2), then read another 256 MiB buffer, so the lines the write left dirty are written
    back now rather than by the timed call's first evictions. The call starts cold and clean."""

    def __init__(self, torch, dev, nbytes=L2_FLUSH_BYTES):
        self.dirty = torch.empty(nbytes // 4, dtype=torch.float32, device=dev)
        self.clean = torch.ones(nbytes // 4, dtype=torch.float32, device=dev)

    def fill_(self, value):
        self.dirty.fill_(value)
        self.clean.sum()
        return self

    describe = "flushed before every step: 256 MiB written, then 256 MiB read (cold, clean L2)"


def hold_device(torch, n):
    """Keeps the device busy (a spin kernel of about 0.2 ms per step to come, at most 20 ms)
    while the host queues the next n steps, so that no host-side delay between a step's
    start event and its launch (Python, the binding, a clock sample) lands inside the timed
    window: every step then starts as soon as the previous work on the stream ends."""
    sleep = getattr(torch.cuda, "_sleep", None)
    if sleep is not None:
        sleep(int(min(2e8, 4e5 * n + 1e6)))   # cycles, ~2 GHz


def time_steps(torch, stream, step, n, flush, restore=None):
    """Runs `step` n times, each after an L2 flush (and `restore`, e.g. C <- C0), and returns
    each call's device time in ms (CUDA events on `stream` around the call only)."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    hold_device(torch, n)
    for i in range(n):
        flush.fill_(float(i))
        if restore is not None:
            restore()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in zip(starts, ends)]


def simt_peak_tflops(sms, mhz=BOOST_MHZ):
    return sms * mhz * 1e6 * FMA_PER_CLK_PER_SM * 2 / 1e12


def tf32_peak():
    """(TF32 dense peak in TFLOP/s, basis): the measured bf16 burst peak scaled by the nominal
    TF32:BF16 ratio, else the nominal TF32 rate."""
    peaks = measured_peaks()
    if peaks.get("bf16_tflops"):
        return (peaks["bf16_tflops"] * TF32_NOMINAL_TFLOPS / BF16_NOMINAL_TFLOPS,
                f"measured bf16 {peaks['bf16_tflops']} TFLOP/s x nominal TF32:BF16 "
                f"{TF32_NOMINAL_TFLOPS:g}:{BF16_NOMINAL_TFLOPS:g} (of measured)")
    return TF32_NOMINAL_TFLOPS, "nominal dense TF32 rate (no measured peak file: of fallback)"


def tensor_roofline(path, achieved_tflops, workload, sms):
    products = 3 if path == "3xtf32" else 1
    peak, basis = tf32_peak()
    kernel = {"3xtf32": "tf32x3_tcgen05", "tf32": "tf32_tcgen05"}[path]
    return {"bound": "tensor", "achieved": round(achieved_tflops, 3), "peak": round(peak, 1),
            "unit": "TFLOP/s", "frac": round(achieved_tflops / peak, 4),
            "issued_tflops": round(products * achieved_tflops, 3),
            "issued_frac": round(products * achieved_tflops / peak, 4),
            "traffic": ncu_traffic(kernel, workload, "3xtf32"),
            "peak_basis": basis + f"; achieved counts 2MNK, issued counts the {products} "
                                  "TF32 product(s) per multiply-add",
            "frac_of_fp32_simt_peak": round(achieved_tflops / simt_peak_tflops(sms), 4)}


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
    entries = {"simt": sg.sgemm, "3xtf32": sg.sgemm_3xtf32, "tf32": sg.sgemm_tf32}
    entry = entries[args.path]

    A_h, B_h, C_h = host_inputs(w)
    A = torch.from_numpy(A_h).to(dev)
    B = torch.from_numpy(B_h).to(dev)
    C = torch.from_numpy(C_h).to(dev)
    C0 = C.clone() if beta != 0.0 else None
    flush = L2Flush(torch, dev)
    stream = torch.cuda.current_stream(dev)
    cfg_id = sg.sgemm_select_config(M, N, K, alpha, A, K, B, N, C, N)
    kernel = (sg.sgemm_config_name(cfg_id) if args.path == "simt"
              else {"3xtf32": "tf32x3_tcgen05", "tf32": "tf32_tcgen05"}[args.path])
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    uuid = getattr(props, "uuid", None)
    uuid = f"GPU-{uuid}" if uuid and not str(uuid).startswith("GPU-") else (str(uuid) if uuid else None)
    restore = (lambda: C.copy_(C0)) if C0 is not None else None

    def step():
        entry(M, N, K, alpha, A, K, B, N, beta, C, N, stream)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        if restore:
            restore()
        step()
    torch.cuda.synchronize(dev)
    if sg.sgemm_device_status(stream) != sg.SGEMM_OK:
        raise RuntimeError(f"device status after warm-up: {sg.sgemm_last_error()}")

    # ---- the timed region: exactly `steps` calls ----
    barrier(dist)
    torch.cuda.synchronize(dev)
    with ClockSampler(local, period_ms=20) as smi, NvmlClocks(uuid, local) as nv:
        wall0 = time.perf_counter()
        step_ms = time_steps(torch, stream, step, args.steps, flush, restore)
        wall = time.perf_counter() - wall0
    barrier(dist)
    if sg.sgemm_device_status(stream) != sg.SGEMM_OK:
        raise RuntimeError(f"device status after timing: {sg.sgemm_last_error()}")
    result_host = C.cpu().numpy() if rank == 0 and not args.no_cpu_baseline else None
    total_ms = max_over_ranks(sum(step_ms), dist, dev)
    value = flops * args.steps * world / (total_ms / 1e3) / 1e9
    clk = merge_clocks(nv.summary(), smi.summary())

    # ---- the same step for at least a second: the clock the kernel sustains ----
    sustained = None
    if not args.no_sustained:
        with ClockSampler(local, period_ms=20) as smi2, NvmlClocks(uuid, local, 0.01) as nv2:
            t0, ms_all = time.perf_counter(), []
            while time.perf_counter() - t0 < args.sustain_s:
                ms_all += time_steps(torch, stream, step, args.steps, flush, restore)
        c2 = merge_clocks(nv2.summary(), smi2.summary())
        sustained = {"steps": len(ms_all), "seconds": round(time.perf_counter() - t0, 3),
                     "value": round(flops * len(ms_all) / (sum(ms_all) / 1e3) / 1e9, 1),
                     "unit": UNIT, "clocks": c2}

    peak_boost = simt_peak_tflops(sms)
    avg_ms = sum(step_ms) / len(step_ms)
    achieved_tflops = flops / (avg_ms / 1e3) / 1e12
    if args.path == "simt":
        roof = {"bound": "alu", "achieved": round(achieved_tflops, 3), "peak": round(peak_boost, 3),
                "unit": "TFLOP/s", "frac": round(achieved_tflops / peak_boost, 4),
                "traffic": ncu_traffic(kernel, args.workload, "simt"),
                "peak_basis": f"{sms} SMs x {BOOST_MHZ:.0f} MHz x {FMA_PER_CLK_PER_SM} FMA/clk x 2"}
        if clk.get("sm_mhz"):
            roof["frac_at_run_clock"] = round(achieved_tflops / simt_peak_tflops(sms, clk["sm_mhz"]), 4)
            roof["run_clock_basis"] = f"median of {clk['samples']} {clk['source']} samples"
    else:
        roof = tensor_roofline(args.path, achieved_tflops, args.workload, sms)

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
                   "l2": L2Flush.describe,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "gflops_median": round(flops / (statistics.median(step_ms) / 1e3) / 1e9, 1),
        "gflops_best": round(flops / (min(step_ms) / 1e3) / 1e9, 1),
        "pct_fp32_simt_peak_boost": round(100.0 * value / world / (peak_boost * 1e3), 2),
        "roofline": roof,
        "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
        "clock_samples": clk["samples"],
        "clock_source": clk["source"],
        "clock_samples_smi": clk["smi_samples"],
        "sustained": sustained,
        "gpu_launches": args.steps * launches_per_call(args.path, kernel, w),
        "wall_s_timed_loop": round(wall, 4),
        "e2e": e2e,
        "device": props.name, "sms": sms,
    }
    if rank == 0 and not args.no_cublas_context:
        line["context_cublas"] = cublas_context(torch, stream, w, A, B, C0 if C0 is not None else C,
                                                flush, max(3, args.warmup), min(args.steps, 50),
                                                value / world)
    if rank == 0 and args.path == "simt" and not args.no_paths:
        line["paths"] = measure_paths(args, torch, sg, stream, w, A, B, C, restore, flush, sms)
    if rank == 0 and not args.no_sweep:
        del A, B, C, C0
        torch.cuda.empty_cache()
        line["sweep"] = measure_sweep(torch, sg, dev, stream, flush, sms, args.sweep_steps)
    if rank == 0 and not args.no_cpu_baseline:
        gf, dt, nrows, threads, check = oracle_sample(w, args.cpu_seconds, A_h, B_h, C_h,
                                                      result=result_host)
        line["cpu_baseline"] = {"value": round(gf, 3), "unit": UNIT, "cores": threads,
                                "kind": "oracle",
                                "sample": f"{nrows} of {M} result rows (all N columns, full K), "
                                          f"{dt:.1f} s, fp64 triple loop, OpenMP over rows"}
        gf1, dt1, n1, _, _ = oracle_sample(w, args.cpu_seconds / 4, A_h, B_h, C_h, threads=1)
        line["cpu_baseline"]["single_core"] = {
            "value": round(gf1, 3), "unit": UNIT, "cores": 1,
            "sample": f"{n1} of {M} result rows (all N columns, full K), {dt1:.1f} s"}
        line["check"] = check
        if not args.no_oracle_sizes:
            line["cpu_baseline"]["sizes"] = oracle_sizes()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    if rank == 0 and line.get("check") and not line["check"]["ok"]:
        raise SystemExit(f"the timed result differs from the oracle: {line['check']}")


def measure_paths(args, torch, sg, stream, w, A, B, C, restore, flush, sms):
    """The tensor-core paths on the bench's workload, under the same timing rules."""
    M, N, K, alpha, beta = w["M"], w["N"], w["K"], w["alpha"], w["beta"]
    flops = 2.0 * M * N * K
    out = {}
    for path, entry in (("3xtf32", sg.sgemm_3xtf32), ("tf32", sg.sgemm_tf32)):
        def step(entry=entry):
            entry(M, N, K, alpha, A, K, B, N, beta, C, N, stream)
        for _ in range(3):
            flush.fill_(1.0)
            if restore:
                restore()
            step()
        ms = time_steps(torch, stream, step, max(3, min(args.steps, 20)), flush, restore)
        if sg.sgemm_device_status(stream) != sg.SGEMM_OK:
            raise RuntimeError(f"device status after the {path} path: {sg.sgemm_last_error()}")
        avg = sum(ms) / len(ms)
        tflops = flops / (avg / 1e3) / 1e12
        kernel = {"3xtf32": "tf32x3_tcgen05", "tf32": "tf32_tcgen05"}[path]
        out[path] = {"value": round(tflops * 1e3, 1), "unit": UNIT, "ms_per_step": round(avg, 4),
                     "steps": len(ms), "kernel": kernel,
                     "gpu_launches_per_call": launches_per_call(path, kernel, w),
                     "roofline": tensor_roofline(path, tflops, args.workload, sms)}
    return out


def size_matched_copy(torch, dev, stream, flush, nbytes, n):
    """The HBM roof for a call that reads `nbytes`, under the same flush and events: a device
    copy (the measured peak's method) that reads the same bytes, nbytes into nbytes. At tens
    of MB the launch and ramp of any kernel are a large part of the time; a copy that reads
    only half the bytes would understate the roof for reads, since the L2 (write-back, 129 MB)
    absorbs its writes during the call."""
    src = torch.ones(max(1, nbytes // 4), dtype=torch.float32, device=dev)
    dst = torch.empty_like(src)
    for _ in range(2):
        flush.fill_(1.0)
        dst.copy_(src)
    ms = time_steps(torch, stream, lambda: dst.copy_(src), n, flush)
    avg = sum(ms) / len(ms)
    return {"ms": round(avg, 4), "read_gbs": round(4 * src.numel() / (avg / 1e3) / 1e9, 1),
            "how": "torch copy reading the call's bytes into another buffer, same flush and events"}


SWEEP = ([f"sweep{n}" for n in (128, 256, 512, 1024, 2048, 4096, 8192, 16384)] +
         ["edge0", "edge1", "edge2", "edge3", "llm_qkv", "llm_up", "llm_down", "llm_head"])


def measure_sweep(torch, sg, dev, stream, flush, sms, steps):
    """GFLOP/s of the SIMT path (and of cuBLAS SGEMM, TF32 off, beside it) on every sweep,
    edge and LLM workload: a few steps each, L2 flushed before every call, CUDA events."""
    peak = simt_peak_tflops(sms)
    rows = []
    for name in SWEEP:
        w = WORKLOADS[name]
        M, N, K, alpha, beta = w["M"], w["N"], w["K"], w["alpha"], w["beta"]
        flops = 2.0 * M * N * K
        A, B, C = device_inputs(torch, dev, w)
        C0 = C.clone() if beta != 0.0 else None
        restore = (lambda: C.copy_(C0)) if C0 is not None else None
        cfg = sg.sgemm_config_name(sg.sgemm_select_config(M, N, K, alpha, A, K, B, N, C, N))

        def step():
            sg.sgemm(M, N, K, alpha, A, K, B, N, beta, C, N, stream)
        for _ in range(2):
            flush.fill_(1.0)
            step()
        n = steps if flops < 2e12 else max(3, steps // 2)
        ms = time_steps(torch, stream, step, n, flush, restore)
        if sg.sgemm_device_status(stream) != sg.SGEMM_OK:
            raise RuntimeError(f"device status after sweep {name}: {sg.sgemm_last_error()}")
        avg = sum(ms) / len(ms)
        gf = flops / (avg / 1e3) / 1e9
        cub = cublas_context(torch, stream, w, A, B, C0 if C0 is not None else C, flush, 2, n, gf)
        row = {"workload": workload_name(name, w), "config": cfg, "gflops": round(gf, 1),
               "ms": round(avg, 4), "steps": n,
               "pct_fp32_simt_peak": round(100.0 * gf / (peak * 1e3), 2),
               "cublas_gflops": cub["value"], "ours_over_cublas": cub["ours_over_it"]}
        if min(M, N) <= 8:   # HBM-bound: the bytes of the large operand and of C
            nbytes = 4 * (M * K + K * N + M * N * (2 if beta != 0.0 else 1))
            row["gbs"] = round(nbytes / (avg / 1e3) / 1e9, 1)
            hbm = measured_peaks().get("hbm_gbs")
            if hbm:
                row["pct_hbm_measured"] = round(100.0 * row["gbs"] / hbm, 2)
            row["size_matched_copy"] = size_matched_copy(torch, dev, stream, flush, nbytes, n)
            row["frac_of_size_matched_copy"] = round(row["size_matched_copy"]["ms"] / avg, 4)
        rows.append(row)
        del A, B, C, C0
        torch.cuda.empty_cache()
    return {"path": "simt", "inputs": "device-drawn from torch's seeded generator (seed 0), "
                                      "the workloads' distributions",
            "l2": L2Flush.describe, "rows": rows}


def launches_per_call(path: str, kernel: str, w) -> int:
    """Kernels one library call launches for the bench's operands (lda = K, ldb = N,
    ldc = N, 16-byte-aligned allocations): the tensor paths split (or round) both operands in
    one launch, then run the GEMM. On the SIMT path a repacked configuration first copies the
    operands whose rows TMA cannot read (K or N not a multiple of 4) into aligned storage, in
    one launch; and when C's rows are not 16-byte aligned (N not a multiple of 4), beta != 0
    and the call has at least 2^22 outputs, a tile kernel's product goes to an aligned scratch
    and one more launch applies the epilogue to C (the skinny and small-problem kernels read C
    themselves)."""
    if path in ("3xtf32", "tf32"):
        return 2
    n = 1
    if kernel.startswith("packed") and (w["K"] % 4 != 0 or w["N"] % 4 != 0):
        n += 1
    tile_kernel = not kernel.startswith(("skinny", "splitk"))
    if (tile_kernel and w.get("beta", 0.0) != 0.0 and w["N"] % 4 != 0
            and w["M"] * w["N"] >= 1 << 22):
        n += 1
    return n


def cublas_context(torch, stream, w, A, B, Csrc, flush, warmup, steps, ours):
    """The same workload through torch.addmm (cuBLAS SGEMM, TF32 off) under the same timing
    rules (out = alpha * A.B + beta * Csrc into a separate buffer): a comparison bar only,
    never a path of the library."""
    M, N, K, alpha, beta = w["M"], w["N"], w["K"], w["alpha"], w["beta"]
    flops = 2.0 * M * N * K
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    out = torch.empty_like(Csrc)
    try:
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                flush.fill_(1.0)
                torch.addmm(Csrc, A, B, beta=beta, alpha=alpha, out=out)
            ms = time_steps(torch, stream,
                            lambda: torch.addmm(Csrc, A, B, beta=beta, alpha=alpha, out=out),
                            steps, flush)
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    del out
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
    ap.add_argument("--no-paths", action="store_true",
                    help="skip the 3xTF32 / TF32 tensor-core paths on the workload")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the size / edge / LLM-shape sweep of the SIMT path")
    ap.add_argument("--sweep-steps", type=int, default=6, help="timed calls per sweep workload")
    ap.add_argument("--no-sustained", action="store_true",
                    help="skip the one-second sustained loop after the timed steps")
    ap.add_argument("--sustain-s", type=float, default=1.0)
    ap.add_argument("--no-oracle-sizes", action="store_true",
                    help="skip timing the oracle on the square sizes of the sweep")
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
