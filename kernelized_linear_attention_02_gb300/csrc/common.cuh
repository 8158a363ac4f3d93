// common.cuh -- small device helpers shared by the kernels of the library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/linattn.h"

namespace la {

// Counts every kernel the library enqueues (la_launch_count).
void note_launch(int n = 1);

// Everything the launchers need, resolved and validated on the host.
struct Problem {
    int64_t B, T;
    int Hq, Hkv, G, Dk, Dv;
    int io_bf16, out_bf16;
    int fmap, norm, gated;
    int decay_dim;  // gated: decay per key dimension (B, T, Hkv, Dk) instead of per head
    int delta;      // delta rules: S += beta k (x) (v - S^T k) after the decay (recurrence only)
    float eps, scale;
    // (B, T) sequence-validity mask, nonzero = valid; null = every step valid
    const uint8_t* mask = nullptr;
};

// Step t of sequence b is valid (Keras request, Masking).
__device__ __forceinline__ bool step_valid(const uint8_t* mask, int64_t bt) { return !mask || mask[bt] != 0; }

__device__ __forceinline__ float load_in(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float load_in(const __nv_bfloat16* p, int64_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void store_out(float* p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, int64_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

// Feature maps of the Keras request ("Feature maps"), evaluated in float32:
// elu_plus_one: x + 1 for x > 0, exp(x) otherwise (ELU slope 1);
// relu:         max(x, 0) + eps;  none: identity.
template <bool kFast>
__device__ __forceinline__ float phi(int fmap, float x, float eps) {
    if (fmap == LA_FMAP_ELU_PLUS_ONE) return x > 0.f ? x + 1.f : (kFast ? __expf(x) : expf(x));
    if (fmap == LA_FMAP_RELU_EPS) return fmaxf(x, 0.f) + eps;
    return x;
}

}  // namespace la
