// delta_args.h -- workspace layout and arguments of the chunk-parallel tile
// kernels (delta_chunk.cu, perdim_chunk.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace la {
namespace delta {

// Workspace of one chunk (bytes).  Tiles are stored in the shared-memory
// operand layout they are used in (128-byte swizzled K-major rows), so the
// consumer loads them with plain bulk copies.
struct Ws {
    static constexpr size_t kW = 0;        // W as B operand: rows t (64), K = k in 2 blocks of 8 KB; hi, lo
    static constexpr size_t kU = 32768;    // U' fp32 [t][v]
    static constexpr size_t kM = 65536;    // M as A operand: rows k' (128), K = k in 2 blocks of 16 KB; hi, lo
    static constexpr size_t kN = 131072;   // N fp32 [k][v]
    static constexpr size_t kS = 196608;   // start state S^T as A operand: rows v (128), K = k; hi, lo
    static constexpr size_t kG = 262144;   // delta: G_t (64 floats), then the step-validity word (2 floats);
                                           // per key dimension: the transition diagonal e^{G_C[k]} (128 floats)
    static constexpr size_t kChunk = 263168;
};

struct Args {
    int B, T, Hq, Hkv, G, nc;  // nc: chunks per stream
    int gated, beta_per_head, out_bf16;
    float scale;
    const __nv_bfloat16* decay;  // (B, T, Hkv), log space
    const __nv_bfloat16* beta;   // (B, T, Hkv) or (B, T)
    const uint8_t* mask;         // (B, T) or null
    const float* S0;             // (B*Hkv, Dk, Dv) or null (zeros)
    float* S_out;                // (B*Hkv, Dk, Dv) or null
    void* y;                     // (B, T, Hq, Dv)
    uint8_t* ws;
    unsigned* err;
};

}  // namespace delta
}  // namespace la
