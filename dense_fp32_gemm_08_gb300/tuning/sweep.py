"""Measure every candidate configuration of every shape class on this GPU.

    python -m dense_fp32_gemm_08_gb300.tuning.sweep [--out PATH] [--reps N]

Each (shape, configuration) is timed with CUDA events over `reps` calls after 3 warm-up
calls, with a 256 MiB buffer written before every call so each starts with a cold L2
(the bench's rule). Unaligned shapes use lda = K, ldb = N, ldc = N with odd sizes (no TMA).
Writes tuning/measured.json: per class, per configuration, the mean GFLOP/s over the class's
shapes and the per-shape figures, plus the device name and SM count.
"""
from __future__ import annotations

import argparse
import json
import time
from pathlib import Path

HERE = Path(__file__).resolve().parent


def main(argv=None):
    import torch

    import dense_fp32_gemm_08_gb300 as sg
    from dense_fp32_gemm_08_gb300.tuning.classes import CLASSES

    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=str(HERE / "measured.json"))
    ap.add_argument("--reps", type=int, default=10)
    ap.add_argument("--classes", nargs="*", default=None,
                    help="re-measure only these classes, keeping the others from --out")
    args = ap.parse_args(argv)
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    ids = {sg.sgemm_config_name(i): i for i in range(sg.sgemm_num_configs())}
    flush = torch.empty(64 << 20, dtype=torch.float32, device=dev)
    result = {"device": torch.cuda.get_device_name(0),
              "sms": torch.cuda.get_device_properties(0).multi_processor_count,
              "when": time.strftime("%Y-%m-%dT%H:%M:%SZ", time.gmtime()), "classes": {}}
    if args.classes:
        if not Path(args.out).exists():
            ap.error(f"--classes re-measures part of an existing table, and {args.out} is missing")
        kept = json.loads(Path(args.out).read_text())["classes"]
        result["classes"] = {c: v for c, v in kept.items() if c not in args.classes}
    try:
        for cls, (shapes, candidates) in CLASSES.items():
            if args.classes and cls not in args.classes:
                continue
            per_cfg = {}
            for (M, N, K) in shapes:
                A = torch.randn(M, K, device=dev)
                B = torch.randn(K, N, device=dev)
                C = torch.randn(M, N, device=dev)
                for name in candidates:
                    sg.sgemm_force_config(ids[name])
                    chosen = sg.sgemm_select_config(M, N, K, 1.0, A, K, B, N, C, N)
                    if chosen != ids[name]:
                        continue  # this configuration cannot run the shape
                    for _ in range(3):
                        sg.sgemm(M, N, K, 1.0, A, K, B, N, 0.0, C, N)
                    torch.cuda.synchronize()
                    total = 0.0
                    for _ in range(args.reps):
                        flush.fill_(1.0)
                        e0 = torch.cuda.Event(enable_timing=True)
                        e1 = torch.cuda.Event(enable_timing=True)
                        e0.record()
                        sg.sgemm(M, N, K, 1.0, A, K, B, N, 0.0, C, N)
                        e1.record()
                        torch.cuda.synchronize()
                        total += e0.elapsed_time(e1)
                    if sg.sgemm_device_status() != sg.SGEMM_OK:
                        raise RuntimeError(f"{name} on {M}x{N}x{K}: device status")
                    gflops = 2.0 * M * N * K / (total / args.reps / 1e3) / 1e9
                    per_cfg.setdefault(name, {})[f"{M}x{N}x{K}"] = round(gflops, 1)
                del A, B, C
            means = {n: round(sum(v.values()) / len(v), 1) for n, v in per_cfg.items()
                     if len(v) == len(shapes)}
            result["classes"][cls] = {"shapes": [f"{M}x{N}x{K}" for (M, N, K) in shapes],
                                      "gflops": per_cfg, "mean_gflops": means,
                                      "winner": max(means, key=means.get) if means else None}
            print(cls, result["classes"][cls]["winner"], means, flush=True)
    finally:
        sg.sgemm_force_config(-1)
    result["classes"] = {c: result["classes"][c] for c in CLASSES if c in result["classes"]}
    Path(args.out).write_text(json.dumps(result, indent=1) + "\n")


if __name__ == "__main__":
    main()
