// config_table_gen.h: written by tuning/gen_table.py from tuning/measured.json;
// do not edit. Per shape class: the configuration that measured fastest.
#pragma once

namespace sg {

constexpr int kNumShapeClasses = 8;

// Indexed by ShapeClass (config_table.h).
constexpr const char *kClassWinner[kNumShapeClasses] = {
    "splitk_cpasync_64x64",  // aligned_tiny: mean TFLOP/s over 128x128x128, 256x256x256, 512x512x512, 128x64x2048: splitk_cpasync_64x64 4.6, ck_tma_256x128_s4 3.6, ck_tma_128x256_s4 3.6, ck_tma_256x128_k64_s2 3.5, ck_tma_128x256_k64_s2 3.5, sk_tma_ws_256x128_k64_s2 2.7, sk_tma_ws_128x256_k64_s2 2.7, sk_tma_ws_256x128_s4 2.6, sk_tma_ws_128x256_s4 2.5, sk_tma_ws_128x128_s3 2.4, dp_tma_128x128_s3 1.7, dp_tma_128x256_s4 1.0, pdp_tma_ws_128x256_s4 1.0
    "sk_tma_ws_128x256_s4",  // aligned_small: default (not measured)
    "sk_tma_ws_128x256_s4",  // aligned_medium: default (not measured)
    "dp_tma_128x128_s3",  // aligned_large: default (not measured)
    "splitk_cpasync_64x64",  // unaligned_tiny: mean TFLOP/s over 97x95x513, 127x129x4099, 255x257x253, 511x509x515: splitk_cpasync_64x64 3.6, sk_cpasync_128x256_s4 2.3, packed_ck_tma_128x256_k64_s2 2.2, packed_sk_tma_256x128_k64_s2 2.1, packed_sk_tma_128x256_s4 2.0, packed_dp_tma_128x128_s3 1.3, dp_cpasync_128x128_s3 1.0, dp_cpasync_128x256_s4 0.7
    "packed_sk_tma_128x256_s4",  // unaligned_small: default (not measured)
    "packed_sk_tma_128x256_s4",  // unaligned_medium: default (not measured)
    "packed_dp_tma_128x128_s3",  // unaligned_large: default (not measured)
};

// measured on NVIDIA GB300 (152 SMs), 2026-12-02T18:05:12Z

}  // namespace sg
