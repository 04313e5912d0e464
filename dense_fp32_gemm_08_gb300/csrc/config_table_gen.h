// config_table_gen.h: written by tuning/gen_table.py from tuning/measured.json;
// do not edit. Per shape class: the configuration that measured fastest.
#pragma once

namespace sg {

constexpr int kNumShapeClasses = 8;

// Indexed by ShapeClass (config_table.h).
constexpr const char *kClassWinner[kNumShapeClasses] = {
    "splitk_cpasync_64x64",  // aligned_tiny: mean TFLOP/s over 128x128x128, 256x256x256, 512x512x512, 128x64x2048: splitk_cpasync_64x64 4.6, ck_tma_256x128_s4 3.6, ck_tma_128x256_s4 3.6, ck_tma_256x128_k64_s2 3.5, ck_tma_128x256_k64_s2 3.5, sk_tma_ws_256x128_k64_s2 2.7, sk_tma_ws_128x256_k64_s2 2.7, sk_tma_ws_256x128_s4 2.6, sk_tma_ws_128x256_s4 2.5, sk_tma_ws_128x128_s3 2.4, dp_tma_128x128_s3 1.7, dp_tma_128x256_s4 1.0, pdp_tma_ws_128x256_s4 1.0
    "sk_tma_ws_128x256_k64_s2",  // aligned_small: mean TFLOP/s over 1024x1024x1024, 1024x2048x1024, 2048x2048x2048: sk_tma_ws_128x256_k64_s2 50.6, sk_tma_ws_256x128_k64_s2 50.5, sk_tma_ws_256x128_s4 49.5, sk_tma_ws_128x256_s4 49.4, ck_tma_128x256_k64_s2 47.5, ck_tma_256x128_k64_s2 47.4, sk_tma_ws_128x128_s3 47.3, ck_tma_256x128_s4 46.8, ck_tma_128x256_s4 46.7, dp_tma_128x128_s3 40.1, splitk_cpasync_64x64 34.4, dp_tma_128x256_s4 31.9, pdp_tma_ws_128x256_s4 30.0
    "sk_tma_ws_256x128_k64_s2",  // aligned_medium: mean TFLOP/s over 4096x4096x4096, 4096x3072x2048, 3072x4096x4096: sk_tma_ws_256x128_k64_s2 64.9, sk_tma_ws_128x256_k64_s2 64.9, sk_tma_ws_256x128_s4 62.8, sk_tma_ws_128x256_s4 62.6, sk_tma_ws_128x128_s3 59.6, dp_tma_128x128_s3 58.3, dp_tma_128x256_s4 56.2, pdp_tma_ws_128x256_s4 53.2, splitk_cpasync_64x64 42.1
    "dp_tma_128x128_s3",  // aligned_large: mean TFLOP/s over 8192x8192x8192, 16384x12288x4096: dp_tma_128x128_s3 67.5, sk_tma_ws_256x128_k64_s2 66.1, sk_tma_ws_128x256_k64_s2 65.9, dp_tma_128x256_s4 65.5, sk_tma_ws_256x128_s4 63.8, sk_tma_ws_128x256_s4 63.6, pdp_tma_ws_128x256_s4 62.0, sk_tma_ws_128x128_s3 60.3, splitk_cpasync_64x64 47.3
    "splitk_cpasync_64x64",  // unaligned_tiny: mean TFLOP/s over 97x95x513, 127x129x4099, 255x257x253, 511x509x515: splitk_cpasync_64x64 3.6, sk_cpasync_128x256_s4 2.3, packed_ck_tma_128x256_k64_s2 2.2, packed_sk_tma_256x128_k64_s2 2.1, packed_sk_tma_128x256_s4 2.0, packed_dp_tma_128x128_s3 1.3, dp_cpasync_128x128_s3 1.0, dp_cpasync_128x256_s4 0.7
    "packed_sk_tma_256x128_k64_s2",  // unaligned_small: mean TFLOP/s over 1001x999x1003, 2047x2045x2049: packed_sk_tma_256x128_k64_s2 40.7, packed_sk_tma_128x256_s4 40.2, packed_ck_tma_128x256_k64_s2 38.6, sk_cpasync_128x256_s4 33.0, packed_dp_tma_128x128_s3 32.8, dp_cpasync_128x256_s4 22.8, dp_cpasync_128x128_s3 22.6, splitk_cpasync_64x64 19.0
    "packed_sk_tma_256x128_k64_s2",  // unaligned_medium: mean TFLOP/s over 4095x3001x1537, 4097x4093x4099: packed_sk_tma_256x128_k64_s2 55.2, packed_sk_tma_128x256_s4 55.1, packed_dp_tma_128x128_s3 54.7, sk_cpasync_128x256_s4 41.7, dp_cpasync_128x128_s3 37.3, dp_cpasync_128x256_s4 36.6, splitk_cpasync_64x64 24.6
    "packed_dp_tma_128x128_s3",  // unaligned_large: mean TFLOP/s over 8191x8193x8195: packed_dp_tma_128x128_s3 63.6, packed_sk_tma_256x128_k64_s2 63.0, packed_sk_tma_128x256_s4 60.2, dp_cpasync_128x256_s4 43.7, sk_cpasync_128x256_s4 43.2, dp_cpasync_128x128_s3 41.9, splitk_cpasync_64x64 26.2
};

// measured on NVIDIA GB300 (152 SMs), 2026-12-02T18:05:12Z

}  // namespace sg
