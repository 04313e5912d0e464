"""Write csrc/config_table_gen.h from tuning/measured.json (run by the build).

The header holds, per shape class, the configuration name that measured fastest and the
measured means as comments; config_table.h maps a problem to its class and looks the name up
in the configuration list. Without a measurement file the header keeps the defaults below.
"""
from __future__ import annotations

import json
from pathlib import Path

HERE = Path(__file__).resolve().parent
MEASURED = HERE / "measured.json"
OUT = HERE.parent / "csrc" / "config_table_gen.h"

DEFAULTS = {
    "aligned_tiny": "dp_tma_128x128_s3", "aligned_small": "sk_tma_ws_128x256_s4",
    "aligned_medium": "sk_tma_ws_128x256_s4", "aligned_large": "dp_tma_128x128_s3",
    "unaligned_tiny": "packed_sk_tma_128x256_s4", "unaligned_small": "packed_sk_tma_128x256_s4",
    "unaligned_medium": "packed_sk_tma_128x256_s4", "unaligned_large": "packed_dp_tma_128x128_s3",
}


def render(measured: dict | None) -> str:
    from dense_fp32_gemm_08_gb300.tuning.classes import CLASS_ORDER
    lines = ["// config_table_gen.h: written by tuning/gen_table.py from tuning/measured.json;",
             "// do not edit. Per shape class: the configuration that measured fastest.",
             "#pragma once", "", "namespace sg {", "",
             f"constexpr int kNumShapeClasses = {len(CLASS_ORDER)};", "",
             "// Indexed by ShapeClass (config_table.h).",
             "constexpr const char *kClassWinner[kNumShapeClasses] = {"]
    for cls in CLASS_ORDER:
        winner = DEFAULTS[cls]
        note = "default (not measured)"
        if measured and measured.get("classes", {}).get(cls, {}).get("winner"):
            c = measured["classes"][cls]
            winner = c["winner"]
            means = ", ".join(f"{k} {v / 1000:.1f}" for k, v in
                              sorted(c["mean_gflops"].items(), key=lambda kv: -kv[1]))
            note = f"mean TFLOP/s over {', '.join(c['shapes'])}: {means}"
        lines.append(f"    \"{winner}\",  // {cls}: {note}")
    lines += ["};", ""]
    if measured:
        lines.append(f"// measured on {measured.get('device')} ({measured.get('sms')} SMs), "
                     f"{measured.get('when')}")
    lines += ["", "}  // namespace sg", ""]
    return "\n".join(lines)


def generate() -> Path:
    measured = json.loads(MEASURED.read_text()) if MEASURED.exists() else None
    text = render(measured)
    if not OUT.exists() or OUT.read_text() != text:
        OUT.write_text(text)
    return OUT


if __name__ == "__main__":
    print(generate())
