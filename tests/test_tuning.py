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
    for (M, N, K) in shapes:
        cls = classes.classify(M, N, aligned=True)
        assert name(sel(M, N, K, 1.0, FAKE, K, FAKE, N, FAKE, N)) == measured["classes"][cls]["winner"]
    for (M, N, K) in [(97, 95, 513), (1001, 999, 1003), (4095, 3001, 1537), (8191, 8193, 8195)]:
        cls = classes.classify(M, N, aligned=False)
        got = name(sel(M, N, K, 1.0, FAKE, K, FAKE, N, FAKE, N))
        assert got == measured["classes"][cls]["winner"], (M, N, K, cls)


@pytest.mark.parametrize("M,N,aligned,want", [(64, 64, True, "aligned_tiny"),
                                              (4096, 4096, True, "aligned_medium"),
                                              (8192, 8192, False, "unaligned_large"),
                                              (1000, 1000, False, "unaligned_small")])
def test_classify(M, N, aligned, want):
    assert classes.classify(M, N, aligned) == want
