import os
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size problem, minutes of host work")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()


@pytest.fixture(scope="session")
def sgemm_lib():
    """The CUDA library's C ABI (built in-tree on first use if the .so is missing)."""
    import dense_fp32_gemm_08_gb300 as pkg
    if not pkg.library_path().exists():
        from dense_fp32_gemm_08_gb300 import _build
        _build.build()
    return pkg


def _gpu_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _gpu_available() or os.environ.get("SGEMM_FORCE_GPU_TESTS"):
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)
