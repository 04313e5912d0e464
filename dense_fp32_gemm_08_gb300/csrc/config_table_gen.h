// config_table_gen.h: written by tuning/gen_table.py from tuning/measured.json;
// do not edit. Per shape class: the configuration that measured fastest.
#pragma once

namespace sg {

constexpr int kNumShapeClasses = 8;

// Indexed by ShapeClass (config_table.h).
constexpr const char *kClassWinner[kNumShapeClasses] = {
    "sk_tma_ws_128x256_s4",  // aligned_tiny: mean TFLOP/s over 96x96x512, 128x64x2048: sk_tma_ws_128x256_s4 0.5, sk_tma_ws_256x128_s4 0.5, sk_tma_ws_256x128_k64_s2 0.4, sk_tma_ws_128x256_k64_s2 0.4, dp_tma_128x128_s3 0.2, dp_tma_128x256_s4 0.1, pdp_tma_ws_128x256_s4 0.1
    "sk_tma_ws_128x256_s4",  // aligned_small: mean TFLOP/s over 512x512x512, 1024x1024x1024, 2048x2048x2048: sk_tma_ws_128x256_s4 35.2, sk_tma_ws_256x128_s4 35.1, sk_tma_ws_128x256_k64_s2 34.4, sk_tma_ws_256x128_k64_s2 34.3, dp_tma_128x128_s3 25.4, dp_tma_128x256_s4 23.1, pdp_tma_ws_128x256_s4 22.4
    "sk_tma_ws_128x256_k64_s2",  // aligned_medium: mean TFLOP/s over 4096x4096x4096, 4096x3072x2048, 3072x4096x4096: sk_tma_ws_128x256_k64_s2 63.3, sk_tma_ws_256x128_k64_s2 63.3, sk_tma_ws_256x128_s4 62.1, sk_tma_ws_128x256_s4 62.1, dp_tma_128x128_s3 57.3, dp_tma_128x256_s4 54.9, pdp_tma_ws_128x256_s4 52.7
    "dp_tma_128x128_s3",  // aligned_large: mean TFLOP/s over 8192x8192x8192, 16384x12288x4096: dp_tma_128x128_s3 65.9, sk_tma_ws_128x256_k64_s2 64.4, sk_tma_ws_256x128_k64_s2 64.4, dp_tma_128x256_s4 64.0, sk_tma_ws_256x128_s4 63.0, sk_tma_ws_128x256_s4 63.0, pdp_tma_ws_128x256_s4 61.4
    "sk_cpasync_128x256_s4",  // unaligned_tiny: mean TFLOP/s over 97x95x513, 127x129x4099: sk_cpasync_128x256_s4 1.0, packed_sk_tma_128x256_s4 0.9, packed_sk_tma_256x128_k64_s2 0.8, packed_dp_tma_128x128_s3 0.3, dp_cpasync_128x128_s3 0.2, dp_cpasync_128x256_s4 0.1
    "packed_sk_tma_128x256_s4",  // unaligned_small: mean TFLOP/s over 1001x999x1003, 2047x2045x2049: packed_sk_tma_128x256_s4 37.9, packed_sk_tma_256x128_k64_s2 37.6, sk_cpasync_128x256_s4 33.4, packed_dp_tma_128x128_s3 30.1, dp_cpasync_128x128_s3 22.2, dp_cpasync_128x256_s4 22.0
    "packed_sk_tma_128x256_s4",  // unaligned_medium: mean TFLOP/s over 4095x3001x1537, 4097x4093x4099: packed_sk_tma_128x256_s4 54.8, packed_sk_tma_256x128_k64_s2 54.0, packed_dp_tma_128x128_s3 53.3, sk_cpasync_128x256_s4 40.8, dp_cpasync_128x128_s3 36.7, dp_cpasync_128x256_s4 35.9
    "packed_dp_tma_128x128_s3",  // unaligned_large: mean TFLOP/s over 8191x8193x8195: packed_dp_tma_128x128_s3 62.4, packed_sk_tma_256x128_k64_s2 61.5, packed_sk_tma_128x256_s4 59.6, dp_cpasync_128x256_s4 42.8, sk_cpasync_128x256_s4 42.2, dp_cpasync_128x128_s3 41.7
};

// measured on NVIDIA GB300 (152 SMs), 2026-12-02T10:56:48Z

}  // namespace sg
