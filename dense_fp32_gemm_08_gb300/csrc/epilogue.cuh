// epilogue.cuh: the fused epilogue shared by every kernel,
//   D = act(alpha * acc + bias[n]) + beta * C     (C read only when beta != 0),
// with act one of the activations below (their published definitions; the math functions
// are CUDA's own erff / tanhf / expf).
#pragma once

#include <cuda_runtime.h>

namespace sg {

enum Activation : int {
    kActNone = 0,
    kActRelu = 1,      // max(x, 0), NaN stays NaN
    kActGelu = 2,      // 0.5 x (1 + erf(x / sqrt 2))            (Hendrycks & Gimpel 2016)
    kActGeluTanh = 3,  // 0.5 x (1 + tanh(sqrt(2/pi)(x + 0.044715 x^3)))   (same paper)
    kActSilu = 4,      // x / (1 + exp(-x))                      (Elfwing, Uchibe & Doya 2018)
};

__device__ __forceinline__ float activate(float x, int act) {
    switch (act) {
        case kActRelu: return x > 0.0f ? x : (x != x ? x : 0.0f);
        case kActGelu: return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));
        case kActGeluTanh: {
            const float u = 0.79788456080286536f * (x + 0.044715f * x * x * x);
            return 0.5f * x * (1.0f + tanhf(u));
        }
        case kActSilu: return x / (1.0f + expf(-x));
        default: return x;
    }
}

// One output value from an already loaded C value: alpha * acc (+ bias) -> act
// (+ beta * c_value). c_value is ignored when beta == 0.
__device__ __forceinline__ float epilogue_apply(float acc, float alpha, float beta,
                                                const float *bias, int col, int act,
                                                float c_value) {
    float v = alpha * acc;
    if (bias) v += bias[col];
    v = activate(v, act);
    if (beta != 0.0f) v = fmaf(beta, c_value, v);
    return v;
}

// The same, reading C through `c`, which is only dereferenced when beta != 0.
__device__ __forceinline__ float epilogue_value(float acc, float alpha, float beta,
                                                const float *bias, int col, int act,
                                                const float *c) {
    return epilogue_apply(acc, alpha, beta, bias, col, act, beta != 0.0f ? *c : 0.0f);
}

}  // namespace sg
