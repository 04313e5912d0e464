// config_table.h: per-shape-class choice of SIMT kernel configuration.
#pragma once

#include "simt_gemm.cuh"

namespace sg {

// Picks the configuration id for a problem from its shape class and operand alignment.
inline int table_choose(const SimtProblem &p) {
    const bool tma = simt_config_supports(0, p);
    const bool small = static_cast<long long>(p.M) * p.N <= 256LL * 256;
    if (tma) return small ? 2 : 0;
    return small ? 4 : 3;
}

}  // namespace sg
