"""Host-side logic of bench.py without a GPU: argument rules, the clock-sample parser, the
ncu-traffic lookup, the CPU-oracle timer and the max-over-ranks reduction of the replica
runs (two gloo ranks on CPU)."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
sys.path.insert(0, str(ROOT))

import bench  # noqa: E402


def test_defaults_and_argument_rules():
    a = bench.parse([])
    assert a.gpus == 1 and a.impl == "ours" and a.workload == "headline" and a.warmup >= 3
    with pytest.raises(SystemExit):
        bench.parse(["--warmup", "2"])
    w = bench.WORKLOADS["headline"]
    assert (w["M"], w["N"], w["K"], w["alpha"], w["beta"]) == (4096, 4096, 4096, 1.0, 0.0)
    assert 2 * w["M"] * w["N"] * w["K"] == 137_438_953_472
    for name in ("edge0", "edge1", "edge2", "edge3", "llm_qkv", "llm_up", "llm_down",
                 "llm_head", "sweep16384", "sq256_ab"):
        assert name in bench.WORKLOADS


def test_clock_summary_parses_reasons():
    s = bench.ClockSampler(0)
    s.lines = ["2070, 2070, 900.1, 0x0000000000000000",
               "1980, 2070, 1390.0, 0x0000000000000004",
               "2070, 2070, 1200.0, 0x0000000000000000",
               "garbage"]
    out = s.summary()
    assert out["sm_mhz"] == 2070 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"] and out["samples"] == 3
    assert bench.ClockSampler(0).summary()["sm_mhz"] is None


def test_ncu_traffic_requires_matching_source(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    (tmp_path / "profiles").mkdir()
    (tmp_path / "dense_fp32_gemm_08_gb300" / "csrc").mkdir(parents=True)
    src = tmp_path / "dense_fp32_gemm_08_gb300" / "csrc" / "simt_gemm.cu"
    src.write_text("// v1\nint f() { return 1; }\n")
    h = bench.source_hash()
    data = {"kern@headline": {"dram_bytes_per_launch": 123, "source_hash": h}}
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps(data))
    assert bench.ncu_traffic("kern", "headline") == 123
    (tmp_path / "dense_fp32_gemm_08_gb300" / "csrc" / "tf32x3_gemm.cu").write_text("int g;")
    assert bench.ncu_traffic("kern", "headline") == 123  # another path's file: still valid
    src.write_text("/* reworded */\nint f()  {\n  return 1;  // same code\n}\n")
    assert bench.ncu_traffic("kern", "headline") == 123  # comments and layout only: still valid
    src.write_text("// v1\nint f() { return 2; }\n")
    assert bench.ncu_traffic("kern", "headline") is None  # the code changed
    assert bench.ncu_traffic("other", "headline") is None


def test_code_of_drops_comments_only():
    assert bench.code_of("a = 1; // x\n/* y\n z */ b  =\n 2;") == "a = 1; b = 2;"
    assert bench.code_of("x = 1;") != bench.code_of("x = 2;")


def test_oracle_timer_counts_rows():
    import synth
    w = dict(M=64, N=48, K=32, alpha=1.0, beta=0.5, dist="uniform")
    A, B, C = synth.uniform(64, 32, 0), synth.uniform(32, 48, 1), synth.uniform(64, 48, 2)
    t = bench.OracleTimer(w, A, B, C)
    n = t.rows_for(0.001)
    assert 1 <= n <= 64
    dt, rows = t.run(10)
    assert rows == 10 and dt > 0


_CHILD = r"""
import os, sys
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
rank = dist.get_rank()
got = bench.max_over_ranks(float(10 + 5 * rank), dist)
bench.barrier(dist)
print("RESULT", rank, got, flush=True)
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_ranks_gloo_world_size_2():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", _CHILD.format(root=str(ROOT))],
                                      env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                      text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (out, err) in zip(procs, outs):
        assert p.returncode == 0, err
    results = sorted(line.split()[1:] for out, _ in outs for line in out.splitlines()
                     if line.startswith("RESULT"))
    assert results == [["0", "15.0"], ["1", "15.0"]]


def test_reference_arm_runs_on_cpu():
    proc = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference",
                           "--workload", "sq256", "--steps", "3", "--warmup", "3",
                           "--cpu-seconds", "0.5"], capture_output=True, text=True, timeout=300)
    assert proc.returncode == 0, proc.stderr
    line = json.loads(proc.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_oracle_sample_single_core_restores_threads():
    import oracle
    full = oracle.max_threads()
    w = bench.WORKLOADS["sq256"]
    A, B, C = bench.host_inputs(w)
    gf, dt, n, threads, check = bench.oracle_sample(w, 0.05, A, B, C, threads=1)
    assert threads == 1 and gf > 0 and 1 <= n <= w["M"] and check is None
    assert oracle.max_threads() == full


def test_result_check_against_the_oracle_rows():
    # The bench's check compares the timed result with the oracle rows of its CPU sample: an
    # exact result passes, one wrong cell fails it.
    import oracle
    w = bench.WORKLOADS["sq256_ab"]
    A, B, C = bench.host_inputs(w)
    full = oracle.sgemm(256, 256, 256, w["alpha"], A, 256, B, 256, w["beta"], C, 256)
    gf, dt, n, threads, check = bench.oracle_sample(w, 0.05, A, B, C, result=full)
    assert check["ok"] and check["normalized_error"] == 0.0 and check["rows"] >= 1
    bad = full.copy()
    bad[:, 7] += 1.0
    _, _, _, _, check = bench.oracle_sample(w, 0.05, A, B, C, result=bad)
    assert not check["ok"]


def test_merge_clocks_prefers_nvml_and_unions_reasons():
    nv = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 22}
    smi = {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0, "reasons": ["hw_slowdown"], "samples": 2}
    m = bench.merge_clocks(nv, smi)
    assert m["sm_mhz"] == 2070.0 and m["samples"] == 22 and m["source"] == "nvml"
    assert m["reasons"] == ["hw_slowdown", "sw_power_cap"]
    m = bench.merge_clocks({"sm_mhz": None, "samples": 0, "reasons": []}, smi)
    assert m["source"] == "nvidia-smi" and m["sm_mhz"] == 2055.0


def test_nvml_sampler_without_a_driver_reports_no_samples():
    with bench.NvmlClocks(None, 0, 0.001) as nv:
        pass
    assert nv.summary()["samples"] >= 0


def test_launches_per_call():
    edge0 = bench.WORKLOADS["edge0"]  # 4095 x 3001 x 1537, beta = -1.3: repack + GEMM + C pass
    assert bench.launches_per_call("simt", "sk_tma_ws_128x256_k64_s2", bench.WORKLOADS["headline"]) == 1
    assert bench.launches_per_call("simt", "packed_sk_tma_256x128_k64_s2", edge0) == 3
    assert bench.launches_per_call("simt", "packed_sk_tma_256x128_k64_s2", dict(edge0, beta=0.0)) == 2
    small = {"M": 127, "N": 129, "K": 4099, "beta": -1.3}  # under 2^22 outputs: C read in place
    assert bench.launches_per_call("simt", "splitk_cpasync_64x64", small) == 1
    assert bench.launches_per_call("simt", "skinny_wide_m8", bench.WORKLOADS["edge1"]) == 1
    assert bench.launches_per_call("3xtf32", "tf32x3_tcgen05", edge0) == 2


def test_oracle_sizes_are_bounded_and_labelled():
    # Timing the oracle on square sizes: the small ones in full (and on one core), the large
    # ones on a row sample, extrapolated and labelled (small sizes keep this test quick).
    out = bench.oracle_sizes(rows_cap_s=1e-6, sizes=(32, 64, 160), full_up_to=64,
                             single_core_up_to=32)
    assert sorted({r["n"] for r in out}) == [32, 64, 160]
    for r in out:
        assert r["gflops"] > 0 and r["cores"] >= 1 and r["seconds_full"] >= 0
        assert (r["how"] == "full") == (r["n"] <= 64)
    assert [r["cores"] for r in out if r["n"] == 32][-1] == 1
