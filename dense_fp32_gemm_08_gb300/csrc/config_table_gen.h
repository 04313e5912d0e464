// config_table_gen.h: written by tuning/gen_table.py from tuning/measured.json;
// do not edit. Per shape class: the configuration that measured fastest.
#pragma once

namespace sg {

constexpr int kNumShapeClasses = 8;

// Indexed by ShapeClass (config_table.h).
constexpr const char *kClassWinner[kNumShapeClasses] = {
    "sk_tma_ws_128x128_s3",  // aligned_tiny: mean TFLOP/s over 96x96x512, 128x64x2048: sk_tma_ws_128x128_s3 0.6, sk_tma_ws_128x256_s4 0.5, sk_tma_ws_256x128_s4 0.5, sk_tma_ws_128x256_k64_s2 0.5, sk_tma_ws_256x128_k64_s2 0.4, dp_tma_128x128_s3 0.2, dp_tma_128x256_s4 0.1, pdp_tma_ws_128x256_s4 0.1
    "sk_tma_ws_128x256_k64_s2",  // aligned_small: mean TFLOP/s over 512x512x512, 1024x1024x1024, 2048x2048x2048: sk_tma_ws_128x256_k64_s2 36.3, sk_tma_ws_256x128_k64_s2 36.3, sk_tma_ws_256x128_s4 35.5, sk_tma_ws_128x256_s4 35.5, sk_tma_ws_128x128_s3 34.4, dp_tma_128x128_s3 26.4, dp_tma_128x256_s4 23.8, pdp_tma_ws_128x256_s4 22.5
    "sk_tma_ws_256x128_k64_s2",  // aligned_medium: mean TFLOP/s over 4096x4096x4096, 4096x3072x2048, 3072x4096x4096: sk_tma_ws_256x128_k64_s2 65.0, sk_tma_ws_128x256_k64_s2 64.9, sk_tma_ws_256x128_s4 62.8, sk_tma_ws_128x256_s4 62.7, sk_tma_ws_128x128_s3 59.6, dp_tma_128x128_s3 58.3, dp_tma_128x256_s4 56.2, pdp_tma_ws_128x256_s4 53.2
    "dp_tma_128x128_s3",  // aligned_large: mean TFLOP/s over 8192x8192x8192, 16384x12288x4096: dp_tma_128x128_s3 67.5, sk_tma_ws_256x128_k64_s2 66.0, sk_tma_ws_128x256_k64_s2 65.9, dp_tma_128x256_s4 65.5, sk_tma_ws_256x128_s4 63.8, sk_tma_ws_128x256_s4 63.6, pdp_tma_ws_128x256_s4 62.0, sk_tma_ws_128x128_s3 60.2
    "sk_cpasync_128x256_s4",  // unaligned_tiny: mean TFLOP/s over 97x95x513, 127x129x4099: sk_cpasync_128x256_s4 1.0, packed_sk_tma_256x128_k64_s2 1.0, packed_sk_tma_128x256_s4 1.0, packed_dp_tma_128x128_s3 0.3, dp_cpasync_128x128_s3 0.2, dp_cpasync_128x256_s4 0.1
    "packed_sk_tma_256x128_k64_s2",  // unaligned_small: mean TFLOP/s over 1001x999x1003, 2047x2045x2049: packed_sk_tma_256x128_k64_s2 38.6, packed_sk_tma_128x256_s4 38.0, sk_cpasync_128x256_s4 33.8, packed_dp_tma_128x128_s3 31.5, dp_cpasync_128x128_s3 23.0, dp_cpasync_128x256_s4 22.3
    "packed_sk_tma_256x128_k64_s2",  // unaligned_medium: mean TFLOP/s over 4095x3001x1537, 4097x4093x4099: packed_sk_tma_256x128_k64_s2 55.3, packed_sk_tma_128x256_s4 55.2, packed_dp_tma_128x128_s3 54.7, sk_cpasync_128x256_s4 41.7, dp_cpasync_128x128_s3 37.3, dp_cpasync_128x256_s4 36.6
    "packed_dp_tma_128x128_s3",  // unaligned_large: mean TFLOP/s over 8191x8193x8195: packed_dp_tma_128x128_s3 63.7, packed_sk_tma_256x128_k64_s2 63.1, packed_sk_tma_128x256_s4 60.2, dp_cpasync_128x256_s4 43.7, sk_cpasync_128x256_s4 43.2, dp_cpasync_128x128_s3 41.9
};

// measured on NVIDIA GB300 (152 SMs), 2026-12-02T13:30:26Z

}  // namespace sg
