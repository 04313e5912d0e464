"""Builds the CUDA library ``libsgemm_gb300.so`` in-tree for sm_103a.

Every ``csrc/*.cu`` is compiled in parallel with
``nvcc -gencode arch=compute_103a,code=sm_103a -O3 -lineinfo`` and linked with
``nvcc -shared`` (static CUDA runtime). ptxas resource usage (registers, spills, shared
memory per kernel) is kept in ``_build/ptxas.txt``. A rebuild happens only when a source or
header is newer than the library, or when ``force=True``.
"""
from __future__ import annotations

import concurrent.futures
import os
import subprocess
import sys
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD_DIR = PKG / "_build"
LIBRARY = PKG / "libsgemm_gb300.so"
GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH") or "/usr/local/cuda"
    cand = Path(home) / "bin" / "nvcc"
    return str(cand) if cand.exists() else "nvcc"


def _sources() -> list[Path]:
    return sorted(CSRC.glob("*.cu"))


def _inputs() -> list[Path]:
    return _sources() + sorted(CSRC.glob("*.cuh")) + sorted(CSRC.glob("*.h")) + \
        sorted(INCLUDE.glob("*.h")) + [Path(__file__)] + sorted((PKG / "tuning").glob("*.py")) + \
        sorted((PKG / "tuning").glob("*.json"))


def is_stale() -> bool:
    if not LIBRARY.exists():
        return True
    built = LIBRARY.stat().st_mtime
    return any(p.stat().st_mtime > built for p in _inputs())


def _compile(src: Path) -> tuple[Path, str]:
    obj = BUILD_DIR / (src.stem + ".o")
    cmd = [_nvcc(), *GENCODE, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-Xptxas", "-v", f"-I{INCLUDE}", f"-I{CSRC}", "-c", str(src), "-o", str(obj)]
    proc = subprocess.run(cmd, capture_output=True, text=True)
    if proc.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src.name}:\n{proc.stdout}\n{proc.stderr}")
    return obj, proc.stderr


def generate_sources() -> None:
    """Write csrc/config_table_gen.h from the measured tuning data."""
    if str(ROOT) not in sys.path:
        sys.path.insert(0, str(ROOT))
    from dense_fp32_gemm_08_gb300.tuning import gen_table
    gen_table.generate()


def build(force: bool = False, verbose: bool = False) -> Path:
    """Compile and link the library; returns its path."""
    generate_sources()
    if not force and not is_stale():
        return LIBRARY
    BUILD_DIR.mkdir(exist_ok=True)
    srcs = _sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        results = list(ex.map(_compile, srcs))
    report = "\n".join(f"== {src.name}\n{log}" for src, (_, log) in zip(srcs, results))
    (BUILD_DIR / "ptxas.txt").write_text(report)
    if verbose:
        print(report)
    tmp = LIBRARY.with_suffix(".so.tmp")
    cmd = [_nvcc(), *GENCODE, "-shared", "-o", str(tmp)] + [str(o) for o, _ in results]
    proc = subprocess.run(cmd, capture_output=True, text=True)
    if proc.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{proc.stdout}\n{proc.stderr}")
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIBRARY)
