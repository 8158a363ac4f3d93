// chunk_args.h -- parameters of the tensor-core chunk kernel (host + device).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace la {
namespace chunk {

enum Mode { kCausal = 0, kState = 1, kApply = 2 };

// error codes recorded in *err (bit per wait site)
enum : unsigned {
    kErrFullKV = 1u << 0, kErrEmptyKV = 1u << 1, kErrFullQ = 1u << 2, kErrEmptyQ = 1u << 3,
    kErrConvKV = 1u << 4, kErrConvQ = 1u << 5, kErrStateReady = 1u << 6, kErrStateDone = 1u << 7,
    kErrAFull = 1u << 8, kErrAEmpty = 1u << 9, kErrATFull = 1u << 10, kErrATEmpty = 1u << 11,
    kErrYFull = 1u << 12, kErrYEmpty = 1u << 13
};

struct Args {
    int B, T, Hq, Hkv, G;
    int cps;   // chunks per segment
    int nseg;  // segments per (b, kv head)
    int fold_r;  // causal: state-pass increments per segment (the state pass may run on sub-segments)
    int fmap;
    float eps, scale;
    const float* S_init;  // (B*Hkv, Dk, Dv) initial state (causal) or the global state (apply); may be null
    const float* Z_init;  // (B*Hkv, Dk)
    const float* S_seg;   // causal, nseg > 1: (B*Hkv, nseg, Dk, Dv) state increment of each segment
    const float* Z_seg;   // (B*Hkv, nseg, Dk) key-sum increment of each segment
    const float* G_seg;   // (B*Hkv, nseg) log decay of each segment (gated)
    float* S_dst;         // causal: final state (B*Hkv, Dk, Dv) from the last segment; state: (B*Hkv, nseg, Dk, Dv)
    float* Z_dst;
    float* G_dst;                 // state + gated: (B*Hkv, nseg) log decay of each segment
    const __nv_bfloat16* decay;   // (B, T, Hkv)
    const uint8_t* mask;          // (B, T) step validity, nonzero = valid; null = every step valid
    void* y;                      // (B, T, Hq, Dv) output, bf16 or fp32
    unsigned* err;
};

// One launch of the chunk kernel: variant selectors, grid, arguments, tensor maps.
struct Launch {
    int mode;
    bool norm, gated, out_bf16;
    bool pdl;  // launch as a programmatic dependent of the previous kernel on the stream
    dim3 grid;
    Args args;
    CUtensorMap mq, mk, mv;
};

}  // namespace chunk

cudaError_t chunk_run_causal_d64_bf16(const chunk::Launch& L, cudaStream_t st);
cudaError_t chunk_run_causal_d64_f32(const chunk::Launch& L, cudaStream_t st);
cudaError_t chunk_run_causal_d128_bf16(const chunk::Launch& L, cudaStream_t st);
cudaError_t chunk_run_causal_d128_f32(const chunk::Launch& L, cudaStream_t st);
cudaError_t chunk_run_other_d64(const chunk::Launch& L, cudaStream_t st);
cudaError_t chunk_run_other_d128(const chunk::Launch& L, cudaStream_t st);
// the same launchers for calls with a sequence-validity mask
cudaError_t chunk_run_causal_d64_bf16_mask(const chunk::Launch& L, cudaStream_t st);
cudaError_t chunk_run_causal_d64_f32_mask(const chunk::Launch& L, cudaStream_t st);
cudaError_t chunk_run_causal_d128_bf16_mask(const chunk::Launch& L, cudaStream_t st);
cudaError_t chunk_run_causal_d128_f32_mask(const chunk::Launch& L, cudaStream_t st);
cudaError_t chunk_run_other_d64_mask(const chunk::Launch& L, cudaStream_t st);
cudaError_t chunk_run_other_d128_mask(const chunk::Launch& L, cudaStream_t st);

}  // namespace la
