// config_table.h: per-shape-class choice of SIMT kernel configuration.
//
// Problems with one output dimension of at most 8 go to the HBM-streaming kernels (skinny_*),
// and grids small enough for clusters of four or more CTAs to the cluster split-K kernels.
// The rest fall into eight classes: operands TMA can read in place (16-byte aligned rows) or
// not, times the grid depth in waves of 128 x 128 tiles at two CTAs per SM on the device's
// multiprocessors (read at run time; 152 on a GB300):
// tiny (at most 512 x 512 output cells), under one wave, 1 to 6 waves, 6 waves or more. The
// fastest configuration of each class is measured by tuning/sweep.py on representative shapes
// (CUDA events, L2 flushed before every call) and written into config_table_gen.h by
// tuning/gen_table.py at build time, with the measured means beside each winner. A winner
// that cannot run a particular problem (e.g. a broadcast batch that cannot be repacked) falls
// back to a configuration that can.
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
    kCfgSplitK64 = 19,
    kCfgCk128x256k64 = 20,
    kCfgCk256x128k64 = 21,
    kCfgPackedCk128x256k64 = 22,
    kCfgCk128x256s4 = 23,
    kCfgCk256x128s4 = 24,
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

// Multiprocessors assumed when no device can be queried (a host-only configuration query):
// the GB300's count.
constexpr int kDefaultSms = 152;

// Waves of 128 x 128 tiles at two CTAs per SM on a part with `sms` multiprocessors.
inline double waves_128x128(const SimtProblem &p, int sms) {
    const double tiles = static_cast<double>((p.M + 127) / 128) * ((p.N + 127) / 128) * p.batch;
    return tiles / (2.0 * (sms > 0 ? sms : kDefaultSms));
}

inline int shape_class(const SimtProblem &p, bool aligned, int sms) {
    const int base = aligned ? kAlignedTiny : kUnalignedTiny;
    if (static_cast<long long>(p.M) * p.N * p.batch <= 512LL * 512) return base;
    const double w = waves_128x128(p, sms);
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

// Picks the configuration id for a problem on a part with `sms` multiprocessors (0: unknown,
// taken as kDefaultSms): the bandwidth kernels for skinny shapes, else the measured winner of
// the problem's shape class (falling back to a configuration that can run the problem when
// the winner cannot, e.g. a broadcast batch that cannot be repacked).
// Grids that form clusters of four or more CTAs under the cluster split-K schedule: more than
// 512 x 512 output cells, 128 x 256 tiles numbering at most a quarter of the SMs, and at least
// four 64-wide k-tiles. Measured on a GB300 (TFLOP/s, cluster split-K against the class's
// stream-K winner): 1024^3 40.9 / 38.4, 1001 x 999 x 1003 (repacked) 30.2 / 26.6; with
// clusters of two (1024 x 2048 x 1024: 46.6 / 50.7) or one (2048^3: 53.7 / 62.1) stream-K wins.
// Aligned operands take the 32-wide-stage variant (its first stage lands sooner: 1024^3
// 53.9 us against 54.6 us for the 64-wide one).
inline bool clusterk_preferred(const SimtProblem &p, int sms) {
    if (static_cast<long long>(p.M) * p.N * p.batch <= 512LL * 512) return false;
    const long long tiles = static_cast<long long>((p.M + 127) / 128) * ((p.N + 255) / 256) * p.batch;
    return tiles * 4 <= (sms > 0 ? sms : kDefaultSms) && (p.K + 63) / 64 >= 4;
}

inline int table_choose(const SimtProblem &p, int sms) {
    // One output dimension of at most 8: HBM-bound, the bandwidth kernels (any alignment).
    if (simt_config_supports(kCfgSkinnyTall, p)) return kCfgSkinnyTall;
    if (simt_config_supports(kCfgSkinnyWide, p)) return kCfgSkinnyWide;
    const bool tma = simt_config_supports(kCfgDpTma128x128, p);
    if (clusterk_preferred(p, sms)) {
        const int ck = tma ? kCfgCk128x256s4 : kCfgPackedCk128x256k64;
        if (simt_config_supports(ck, p)) return ck;
    }
    const int cls = shape_class(p, tma, sms);
    const int id = config_by_name(kClassWinner[cls]);
    if (id >= 0 && simt_config_supports(id, p)) return id;
    if (tma) return kCfgSkTma128x256;
    return waves_128x128(p, sms) >= 6.0 ? kCfgDpCp128x128 : kCfgSkCp128x256;
}

}  // namespace sg
