// tiles.cuh -- helpers shared by the tile kernels of the delta rules and of
// the per-key-dimension decay (delta_chunk.cu, perdim_chunk.cu): 128-byte
// swizzled operand rows, bf16 hi/lo splits, step words, tensor maps and the
// per-device kernel configuration.
#pragma once

#include <atomic>

#include <cuda_bf16.h>

#include "kernels.h"
#include "tma_host.h"
#include "umma.cuh"

namespace la {
namespace tile {

using namespace umma;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u);
}
// byte offset of 16-byte chunk cc (8 bf16) of row r in a 128-byte swizzled block
__device__ __forceinline__ uint32_t swc(int r, int cc) {
    return static_cast<uint32_t>(r * 128 + (((cc ^ (r & 7))) << 4));
}
// byte offset of bf16 element (r, col) (col < 64) in a 128-byte swizzled block
__device__ __forceinline__ uint32_t swe(int r, int col) { return swc(r, col >> 3) + ((col & 7) << 1); }

__device__ __forceinline__ uint32_t bf2_bits(__nv_bfloat162 h) { return *reinterpret_cast<uint32_t*>(&h); }
// x = hi + lo, hi = bf16(x), lo = bf16(x - hi), for a pair
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(h);
    hi = bf2_bits(h);
    lo = bf2_bits(__floats2bfloat162_rn(x0 - hf.x, x1 - hf.y));
}
// hi and lo parts of 8 values as two 16-byte words
__device__ __forceinline__ void split8(const float* f, uint4& hi, uint4& lo) {
    split2(f[0], f[1], hi.x, lo.x);
    split2(f[2], f[3], hi.y, lo.y);
    split2(f[4], f[5], hi.z, lo.z);
    split2(f[6], f[7], hi.w, lo.w);
}
__device__ __forceinline__ void st16(uint8_t* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

// 64-bit word from the flags of steps 2 lane (even) and 2 lane + 1 (odd);
// warp-collective
__device__ __forceinline__ uint64_t step_word(bool even, bool odd) {
    auto spread = [](uint64_t x) {  // bit i -> bit 2i
        x = (x | (x << 16)) & 0x0000FFFF0000FFFFull;
        x = (x | (x << 8)) & 0x00FF00FF00FF00FFull;
        x = (x | (x << 4)) & 0x0F0F0F0F0F0F0F0Full;
        x = (x | (x << 2)) & 0x3333333333333333ull;
        x = (x | (x << 1)) & 0x5555555555555555ull;
        return x;
    };
    const uint32_t e = __ballot_sync(0xffffffffu, even), o = __ballot_sync(0xffffffffu, odd);
    return spread(e) | (spread(o) << 1);
}

// (D, H, T, B) view of a bf16 activation, 64 x 64 boxes, 128-byte swizzle
inline bool act_map(CUtensorMap* m, const void* base, int H, int64_t T, int64_t B, int D = 128) {
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)H, (uint64_t)T, (uint64_t)B};
    const uint64_t str[3] = {(uint64_t)D * 2, (uint64_t)H * D * 2, (uint64_t)T * H * D * 2};
    const uint32_t box[4] = {64, 1, 64, 1};
    return make_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, 4, dims, str, box,
                           CU_TENSOR_MAP_SWIZZLE_128B);
}

// Raises the dynamic shared-memory limit of a kernel once per device and
// context.
template <typename K>
cudaError_t configure(K kern, int bytes, std::atomic<uint64_t>* flags) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    const uint64_t ctx = current_context_id();
    if (ctx == 0 || flags[dev].load(std::memory_order_acquire) != ctx) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        flags[dev].store(current_context_id(), std::memory_order_release);
    }
    return cudaSuccess;
}


}  // namespace tile
}  // namespace la
