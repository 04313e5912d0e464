// config_table.h: per-shape-class choice of SIMT kernel configuration.
//
// The winner of each shape class is measured (tuning/sweep.py) and written into
// config_table_gen.h by tuning/gen_table.py at build time. Earlier hand sweeps that shaped the
// classes (bench.py with SGEMM_FORCE_CONFIG, one configuration at a time, GB300, 152 SMs):
//
//   class                       measured                                         choice
//   aligned, <  6 waves of       4096^3: sk 128x256 63.6 TF/s, dp 128x128 62.0,   sk_tma_ws_128x256_s4
//     128x128 tiles at 2/SM      dp 128x256 54.5; 2048^3: sk 128x256 60.5,
//                                dp 128x128 48.2, dp 128x256 53.0
//   aligned, >= 6 waves          8192^3: dp 128x128 65.2, sk 128x256 64.1;         dp_tma_128x128_s3
//                                16384x12288x4096: dp 128x128 65.3, sk 62.7
//   aligned, one tile or less    256^3 and below: latency bound, a single          dp_tma_128x128_s3
//                                128x128 CTA per tile has the shortest chain
//   unaligned (no TMA)           4095x3001x1537: dp cp.async 128x256 30.1 TF/s,    packed_sk_tma_128x256_s4
//                                sk cp.async 128x256 35.2; 127x129x4099: dp        (packed_dp_tma_128x128_s3
//                                cp.async 0.72 ms, sk cp.async 0.10 ms             at >= 6 waves)
//   unaligned, broadcast batch   operands that cannot be repacked once             sk_cpasync_128x256_s4
//   N <= 8 (any alignment)       4096x1x4096: tile kernels 0.55 ms (HBM-bound)     skinny_tall_n8
//   M <= 8 (any alignment)       1x4096x4096: tile kernels 0.34 ms (HBM-bound)     skinny_wide_m8
#pragma once

#include "config_table_gen.h"
#include "simt_gemm.cuh"

namespace sg {

enum : int {
    kCfgDpTma128x256 = 0,
    kCfgDpTma256x128 = 1,
    kCfgDpTma128x128 = 2,
    kCfgDpCp128x256 = 3,
    kCfgDpCp128x128 = 4,
    kCfgSkTma128x256 = 5,
    kCfgPdpTma128x256 = 6,
    kCfgSkTma256x128 = 7,
    kCfgSkTma128x128s3 = 8,
    kCfgSkTma128x128s4 = 9,
    kCfgSkinnyTall = 10,
    kCfgSkinnyWide = 11,
    kCfgSkCp128x256 = 12,
    kCfgSkCp256x128 = 13,
    kCfgPackedSk128x256 = 14,
    kCfgPackedDp128x128 = 15,
    kCfgSkTma128x256k64 = 16,
    kCfgSkTma256x128k64 = 17,
    kCfgPackedSk256x128k64 = 18,
};

// Shape classes, in the order of kClassWinner (config_table_gen.h) and of
// tuning/classes.py, which defines the same rule.
enum ShapeClass : int {
    kAlignedTiny = 0,
    kAlignedSmall,
    kAlignedMedium,
    kAlignedLarge,
    kUnalignedTiny,
    kUnalignedSmall,
    kUnalignedMedium,
    kUnalignedLarge,
};

// Waves of 128 x 128 tiles at two CTAs per SM on a 152-SM part.
inline double waves_128x128(const SimtProblem &p) {
    const double tiles = static_cast<double>((p.M + 127) / 128) * ((p.N + 127) / 128) * p.batch;
    return tiles / (2.0 * 152.0);
}

inline int shape_class(const SimtProblem &p, bool aligned) {
    const int base = aligned ? kAlignedTiny : kUnalignedTiny;
    if (static_cast<long long>(p.M) * p.N * p.batch <= 128LL * 128) return base;
    const double w = waves_128x128(p);
    return base + (w < 1.0 ? 1 : w < 6.0 ? 2 : 3);
}

inline int config_by_name(const char *name) {
    for (int i = 0; i < simt_num_configs(); ++i) {
        const char *a = simt_config(i).name;
        int j = 0;
        while (a[j] && a[j] == name[j]) ++j;
        if (a[j] == name[j]) return i;
    }
    return -1;
}

// Picks the configuration id for a problem: the bandwidth kernels for skinny shapes, else
// the measured winner of the problem's shape class (falling back to a configuration that
// can run the problem when the winner cannot, e.g. a broadcast batch that cannot be
// repacked).
inline int table_choose(const SimtProblem &p) {
    // One output dimension of at most 8: HBM-bound, the bandwidth kernels (any alignment).
    if (simt_config_supports(kCfgSkinnyTall, p)) return kCfgSkinnyTall;
    if (simt_config_supports(kCfgSkinnyWide, p)) return kCfgSkinnyWide;
    const bool tma = simt_config_supports(kCfgDpTma128x128, p);
    const int cls = shape_class(p, tma);
    const int id = config_by_name(kClassWinner[cls]);
    if (id >= 0 && simt_config_supports(id, p)) return id;
    if (tma) return kCfgSkTma128x256;
    return waves_128x128(p) >= 6.0 ? kCfgDpCp128x128 : kCfgSkCp128x256;
}

}  // namespace sg
