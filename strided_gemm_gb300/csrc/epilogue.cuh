// Fused epilogue shared by the kernels: out = act(alpha*acc (+ C_old) + D).
//
// The fusion of "PyTorch demystified 3", section "Summary" (the bias term of a
// feed-forward layer added inside the matmul kernel, saving a pass over C and
// a launch), with the activations the pages name: ReLU, GeluTanh and
// GeluExact ("Chapter 09 CUDA backend", section "Elementwise"), the sigmoid
// ("PyTorch demystified 3") and SiLU ("rvllm CUDA path").  D is an addend laid
// out like an operand; zero strides broadcast it, so a per-column bias has
// rsD = 0, csD = 1, bsD = 0.
//
// Rounding order: the product's own epilogue value first (fmaf(alpha, acc,
// C_old) or alpha*acc, exactly as without the fusion), then one fp32 add of D,
// then the activation through the CUDA math library (expf, tanhf, erff).
#pragma once

#include <cstdint>

#include "debug_check.cuh"
#include "internal.h"

namespace sbg {

enum : int {
    kActNone = 0, kActRelu = 1, kActSigmoid = 2, kActSilu = 3, kActGeluTanh = 4, kActGeluErf = 5
};

// One activation, chosen at compile time (for unrolled loops, so that each
// loop carries one function's code).
template <int ACT>
__device__ __forceinline__ float act_fn(float z) {
    if constexpr (ACT == kActRelu) {
        return z > 0.0f ? z : 0.0f;
    } else if constexpr (ACT == kActSigmoid) {
        return 1.0f / (1.0f + expf(-z));
    } else if constexpr (ACT == kActSilu) {
        return z / (1.0f + expf(-z));
    } else if constexpr (ACT == kActGeluTanh) {
        const float kSqrt2OverPi = 0.7978845608028654f;
        return 0.5f * z * (1.0f + tanhf(kSqrt2OverPi * (z + 0.044715f * z * z * z)));
    } else if constexpr (ACT == kActGeluErf) {
        return 0.5f * z * (1.0f + erff(z * 0.7071067811865476f));
    } else {
        return z;
    }
}

// The activation chosen at run time (a warp-uniform branch).
__device__ __forceinline__ float activate(int act, float z) {
    switch (act) {
        case kActRelu: return act_fn<kActRelu>(z);
        case kActSigmoid: return act_fn<kActSigmoid>(z);
        case kActSilu: return act_fn<kActSilu>(z);
        case kActGeluTanh: return act_fn<kActGeluTanh>(z);
        case kActGeluErf: return act_fn<kActGeluErf>(z);
        default: return z;
    }
}

// The fused part for output (b, m, n), applied to the product's epilogue value.
// `status`: the calling kernel's status word (debug bounds checks).
__device__ __forceinline__ float finish(const EpiParams& e, float v, int64_t b, int64_t m,
                                        int64_t n, unsigned int* status) {
    if (e.D) {
        const float* d = e.D + b * e.bsD + m * e.rsD + n * e.csD;
        if (dbg_in_span(e.D, d, e.d_span, status)) v += __ldg(d);
    }
    return activate(e.act, v);
}

}  // namespace sbg
