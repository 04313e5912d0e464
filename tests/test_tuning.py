"""The measured configuration table: the generated header names each class's fastest
configuration from tuning/measured.json, and the library's class rule agrees with the
Python one the sweep uses."""
from __future__ import annotations

import json

import pytest

from dense_fp32_gemm_08_gb300.tuning import classes, gen_table

FAKE = 1 << 20


def test_generated_header_names_the_measured_winners():
    measured = json.loads(gen_table.MEASURED.read_text())
    text = gen_table.render(measured)
    for cls in classes.CLASS_ORDER:
        c = measured["classes"][cls]
        best = max(c["mean_gflops"], key=c["mean_gflops"].get)
        assert c["winner"] == best
        assert f'"{best}",  // {cls}:' in text
    assert gen_table.OUT.read_text() == text, "config_table_gen.h is stale: rebuild"


def test_library_follows_the_class_table(sgemm_lib):
    measured = json.loads(gen_table.MEASURED.read_text())
    sel, name = sgemm_lib.sgemm_select_config, sgemm_lib.sgemm_config_name
    shapes = [(96, 96, 512), (512, 512, 512), (2048, 2048, 2048), (4096, 4096, 4096),
              (4096, 3072, 2048), (8192, 8192, 8192), (16384, 12288, 4096), (300, 9000, 64)]
    winners = {c: v["winner"] for c, v in measured["classes"].items()}
    for (M, N, K) in shapes + [(1024, 1024, 1024), (768, 1536, 512), (1024, 2048, 1024)]:
        want = classes.expected_config(M, N, K, True, winners)
        assert name(sel(M, N, K, 1.0, FAKE, K, FAKE, N, FAKE, N)) == want, (M, N, K)
    for (M, N, K) in [(97, 95, 513), (1001, 999, 1003), (4095, 3001, 1537), (8191, 8193, 8195)]:
        got = name(sel(M, N, K, 1.0, FAKE, K, FAKE, N, FAKE, N))
        assert got == classes.expected_config(M, N, K, False, winners), (M, N, K)


def test_cluster_split_k_rule():
    assert classes.clusterk_preferred(1024, 1024, 1024)          # 32 tiles: clusters of 4
    assert not classes.clusterk_preferred(1024, 2048, 1024)      # 64 tiles: clusters of 2
    assert not classes.clusterk_preferred(512, 512, 512)         # tiny: the one-warp kernel
    assert not classes.clusterk_preferred(1024, 1024, 192)       # three 64-wide k-tiles
    assert classes.clusterk_preferred(1024, 1024, 1024, sms=152)
    assert not classes.clusterk_preferred(1024, 1024, 1024, sms=76)


@pytest.mark.parametrize("M,N,aligned,want", [(64, 64, True, "aligned_tiny"),
                                              (4096, 4096, True, "aligned_medium"),
                                              (8192, 8192, False, "unaligned_large"),
                                              (1000, 1000, False, "unaligned_small")])
def test_classify(M, N, aligned, want):
    assert classes.classify(M, N, aligned) == want


def test_classify_follows_the_sm_count():
    # 4096 x 4096 is 1024 tiles of 128 x 128: 3.4 waves at two CTAs per SM on 152 SMs,
    # 6.7 waves on a 76-SM part (one die), so the same shape changes class.
    assert classes.classify(4096, 4096, True, sms=152) == "aligned_medium"
    assert classes.classify(4096, 4096, True, sms=76) == "aligned_large"
    assert classes.classify(1024, 1024, True, sms=152) == "aligned_small"
    assert classes.classify(1024, 1024, True, sms=16) == "aligned_medium"


def test_library_class_rule_follows_the_sm_count(tmp_path):
    # The header's rule, compiled on the host, classifies the same shape by the SM count it is
    # given (the library passes the current device's multiprocessor count).
    import shutil
    import subprocess
    from pathlib import Path
    root = Path(__file__).resolve().parents[1]
    csrc = root / "dense_fp32_gemm_08_gb300" / "csrc"
    cuda_inc = Path("/usr/local/cuda/include")
    if not (cuda_inc / "cuda_runtime.h").exists() or shutil.which("g++") is None:
        pytest.skip("needs g++ and the CUDA headers")
    src = tmp_path / "cls.cpp"
    src.write_text(
        '#include "config_table.h"\n#include <cstdio>\n'
        "int main() {\n"
        "  sg::SimtProblem p{};\n"
        "  p.M = 4096; p.N = 4096; p.K = 4096; p.batch = 1;\n"
        "  std::printf(\"%d %d %d\\n\", sg::shape_class(p, true, 152), sg::shape_class(p, true, 76),"
        " sg::shape_class(p, true, 0));\n"
        "  return 0;\n}\n")
    exe = tmp_path / "cls"
    subprocess.run(["g++", "-std=c++17", f"-I{csrc}", f"-I{cuda_inc}", str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    order = classes.CLASS_ORDER
    assert [order[int(x)] for x in out] == ["aligned_medium", "aligned_large", "aligned_medium"]
