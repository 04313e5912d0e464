"""The C ABI without a GPU: the library loads, exports every function include/sgemm.h
declares, rejects bad arguments before touching a device, treats degenerate sizes as
no-ops, and its host-side configuration choice follows operand alignment."""
from __future__ import annotations

import ctypes
import re
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
HEADER = ROOT / "include" / "sgemm.h"


def _declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sgemm\w*)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("sgemm", "sgemm_strided_batched", "sgemm_3xtf32",
                     "sgemm_3xtf32_strided_batched", "sgemm_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(sgemm_lib):
    path = sgemm_lib.library_path()
    out = subprocess.run(["nm", "-D", "--defined-only", str(path)], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in _declared_functions() if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    L = ctypes.CDLL(str(path))
    for n in _declared_functions():
        assert hasattr(L, n)


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "use.c"
    src.write_text('#include "sgemm.h"\nint main(void){ return (int)SGEMM_OK; }\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", f"-I{HEADER.parent}", "-c",
                    str(src), "-o", str(tmp_path / "use.o")], check=True)


def test_status_strings(sgemm_lib):
    L = sgemm_lib.lib()
    for code, name in [(0, b"SGEMM_OK"), (1, b"SGEMM_ERR_INVALID_VALUE"), (2, b"SGEMM_ERR_LAUNCH"),
                       (3, b"SGEMM_ERR_TIMEOUT"), (4, b"SGEMM_ERR_UNSUPPORTED")]:
        assert L.sgemm_status_string(code) == name
    assert L.sgemm_status_string(99).startswith(b"SGEMM_")


FAKE = 1 << 20  # a 16-byte aligned non-null address; argument checks never dereference it


@pytest.mark.parametrize("args,why", [
    ((-1, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4), "M, N and K"),
    ((4, -1, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4), "M, N and K"),
    ((4, 4, -1, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4), "M, N and K"),
    ((4, 4, 8, 1.0, FAKE, 7, FAKE, 4, 0.0, FAKE, 4), "lda"),
    ((4, 4, 8, 1.0, FAKE, 8, FAKE, 3, 0.0, FAKE, 4), "ldb"),
    ((4, 4, 8, 1.0, FAKE, 8, FAKE, 4, 0.0, FAKE, 3), "ldc"),
    ((4, 4, 8, 1.0, FAKE, 8, FAKE, 4, 0.0, None, 4), "C is NULL"),
    ((4, 4, 8, 1.0, None, 8, FAKE, 4, 0.0, FAKE, 4), "A or B"),
    ((4, 4, 8, 1.0, FAKE, 8, None, 4, 0.0, FAKE, 4), "A or B"),
    ((4, 4, 0, 1.0, FAKE, 0, FAKE, 4, 0.0, FAKE, 4), "lda"),
])
def test_invalid_arguments(sgemm_lib, args, why):
    L = sgemm_lib.lib()
    for fn in (L.sgemm, L.sgemm_3xtf32):
        st = fn(*args, None)
        assert st == sgemm_lib.SGEMM_ERR_INVALID_VALUE
        assert why in L.sgemm_last_error().decode()


def test_ex_argument_rules(sgemm_lib):
    L = sgemm_lib.lib()
    # transposed A needs lda >= M, transposed B ldb >= K (the accepted minimum is exercised
    # on real device buffers in test_gpu_trans.py: a valid call here would launch kernels)
    bad_lda = (1, 0, 0, 8, 6, 4, 1.0, FAKE, 7, FAKE, 6, 0.0, FAKE, 6, None)
    assert L.sgemm_ex(*bad_lda) == sgemm_lib.SGEMM_ERR_INVALID_VALUE
    assert "transposed" in L.sgemm_last_error().decode()
    bad_ldb = (0, 1, 0, 8, 6, 4, 1.0, FAKE, 4, FAKE, 3, 0.0, FAKE, 6, None)
    assert L.sgemm_ex(*bad_ldb) == sgemm_lib.SGEMM_ERR_INVALID_VALUE
    for bad in ((2, 0, 0), (0, 5, 0), (0, 0, 9)):
        args = bad + (8, 6, 4, 1.0, FAKE, 8, FAKE, 6, 0.0, FAKE, 6, None)
        assert L.sgemm_ex(*args) == sgemm_lib.SGEMM_ERR_INVALID_VALUE


def test_fused_rejects_unknown_activation(sgemm_lib):
    L = sgemm_lib.lib()
    args = (0, 0, 0, 8, 6, 4, 1.0, FAKE, 4, FAKE, 6, 0.0, FAKE, 6, None, 9, None)
    assert L.sgemm_fused(*args) == sgemm_lib.SGEMM_ERR_INVALID_VALUE
    assert "activation" in L.sgemm_last_error().decode()


def test_invalid_batched_arguments(sgemm_lib):
    L = sgemm_lib.lib()
    base = [8, 8, 8, 1.0, FAKE, 8, 64, FAKE, 8, 64, 0.0, FAKE, 8, 64, 2, None]
    bad = dict(batch=(14, -1), strideA=(6, -1), strideC=(13, 63))
    for name, (pos, value) in bad.items():
        args = list(base)
        args[pos] = value
        assert L.sgemm_strided_batched(*args) == sgemm_lib.SGEMM_ERR_INVALID_VALUE, name


def test_degenerate_sizes_are_noops_without_device(sgemm_lib):
    L = sgemm_lib.lib()
    assert L.sgemm(0, 4, 4, 1.0, None, 4, None, 4, 0.0, None, 4, None) == 0
    assert L.sgemm(4, 0, 4, 1.0, None, 4, None, 1, 0.0, None, 1, None) == 0
    assert L.sgemm_strided_batched(4, 4, 4, 1.0, None, 4, 0, None, 4, 0, 0.0, None, 4, 0, 0,
                                   None) == 0


def test_no_device_is_reported(sgemm_lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    L = sgemm_lib.lib()
    st = L.sgemm(4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4, None)
    assert st == sgemm_lib.SGEMM_ERR_UNSUPPORTED


def test_config_table_names(sgemm_lib):
    n = sgemm_lib.sgemm_num_configs()
    assert n >= 4
    names = [sgemm_lib.sgemm_config_name(i) for i in range(n)]
    assert all(names) and len(set(names)) == n
    assert sgemm_lib.sgemm_config_name(n) is None
    assert sgemm_lib.sgemm_config_name(-1) is None


def test_skinny_shapes_select_bandwidth_kernels(sgemm_lib):
    sel = sgemm_lib.sgemm_select_config
    name = sgemm_lib.sgemm_config_name
    assert name(sel(4096, 1, 4096, 1.0, FAKE, 4096, FAKE, 1, FAKE, 1)).startswith("skinny_tall")
    assert name(sel(1, 4096, 4096, 1.0, FAKE, 4096, FAKE, 4096, FAKE, 4096)).startswith("skinny_wide")
    assert name(sel(8, 9, 64, 1.0, FAKE + 4, 64, FAKE, 9, FAKE, 9)).startswith("skinny_wide")
    assert not name(sel(9, 9, 64, 1.0, FAKE, 64, FAKE, 12, FAKE, 12)).startswith("skinny")


def test_selection_follows_alignment(sgemm_lib):
    sel = sgemm_lib.sgemm_select_config
    name = sgemm_lib.sgemm_config_name
    aligned = name(sel(4096, 4096, 4096, 1.0, FAKE, 4096, FAKE, 4096, FAKE, 4096))
    assert "tma" in aligned
    # operands TMA cannot read are repacked (or, failing that, loaded with cp.async)
    assert "packed" in name(sel(4096, 4096, 4096, 1.0, FAKE + 4, 4096, FAKE, 4096, FAKE, 4096))
    assert "packed" in name(sel(4095, 3001, 1537, 1.0, FAKE, 1537, FAKE, 3001, FAKE, 3001))
    # no kernel for degenerate or scale-only calls
    assert sel(0, 4, 4, 1.0, FAKE, 4, FAKE, 4, FAKE, 4) == -1
    assert sel(4, 4, 4, 0.0, FAKE, 4, FAKE, 4, FAKE, 4) == -1
    assert sel(4, 4, 0, 1.0, FAKE, 1, FAKE, 4, FAKE, 4) == -1


def test_force_config(sgemm_lib):
    sel = sgemm_lib.sgemm_select_config
    try:
        n = sgemm_lib.sgemm_num_configs()
        for i in range(n):
            sgemm_lib.sgemm_force_config(i)
            name = sgemm_lib.sgemm_config_name(i)
            if name.startswith("skinny_tall"):
                shape = (512, 3, 512)
            elif name.startswith("skinny_wide"):
                shape = (3, 512, 512)
            else:
                shape = (512, 512, 512)
            M, N, K = shape
            got = sel(M, N, K, 1.0, FAKE, K, FAKE, N, FAKE, N)
            assert got == i, name
        # a forced skinny kernel cannot take a square problem: the table decides instead
        sgemm_lib.sgemm_force_config([i for i in range(n)
                                      if sgemm_lib.sgemm_config_name(i).startswith("skinny")][0])
        assert not sgemm_lib.sgemm_config_name(
            sel(512, 512, 512, 1.0, FAKE, 512, FAKE, 512, FAKE, 512)).startswith("skinny")
        # a TMA configuration cannot take a misaligned operand: the table decides instead
        tma_ids = [i for i in range(n) if sgemm_lib.sgemm_config_name(i).startswith(("dp_tma", "sk_tma"))]
        sgemm_lib.sgemm_force_config(tma_ids[0])
        got = sel(512, 512, 512, 1.0, FAKE + 4, 512, FAKE, 512, FAKE, 512)
        assert sgemm_lib.sgemm_config_name(got).startswith(("packed", "dp_cpasync", "sk_cpasync",
                                                            "splitk_cpasync"))
        with pytest.raises(sgemm_lib.SgemmError):
            sgemm_lib.sgemm_force_config(n)
    finally:
        sgemm_lib.sgemm_force_config(-1)


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path, sgemm_lib):
    monkeypatch.setattr(sgemm_lib, "_LIBRARY", tmp_path / "missing.so")
    monkeypatch.setattr(sgemm_lib, "_lib", None)
    with pytest.raises(RuntimeError):
        sgemm_lib.lib()


class _FailingLibrary:
    """Stands in for the loaded library: every product call fails the way a device-memory
    shortage or a launch error would, with the library's own message."""

    def __init__(self, status, message):
        self.status, self.message = status, message

    def __getattr__(self, name):
        if name == "sgemm_last_error":
            return lambda: self.message
        if name == "sgemm_status_string":
            return lambda status: b"SGEMM_ERR_LAUNCH"
        return lambda *args: self.status


@pytest.mark.parametrize("status,message", [
    (2, b"split-K workspace allocation failed: out of memory"),
    (2, b"kernel launch failed: invalid configuration argument"),
    (3, b""),
])
def test_binding_raises_the_library_error(monkeypatch, sgemm_lib, status, message):
    monkeypatch.setattr(sgemm_lib, "_lib", _FailingLibrary(status, message))
    with pytest.raises(sgemm_lib.SgemmError) as info:
        sgemm_lib.sgemm(4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4)
    assert info.value.status == status
    assert (message.decode() or "SGEMM_ERR_LAUNCH") in str(info.value)
    with pytest.raises(sgemm_lib.SgemmError):
        sgemm_lib.sgemm_3xtf32(4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4)
