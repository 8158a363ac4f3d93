// decode.cu -- one streaming token per sequence, state updated in place.
//
// "Causal Linear Attention": S_i = S_{i-1} + phi(k_i) v_i^T, Z_i = Z_{i-1} +
// phi(k_i), output phi(q_i)^T S_i / (phi(q_i)^T Z_i + eps); ONNX-light
// "LinearAttention" with T = 1 and the gated rule S = exp(g) S + k (x) v.
//
// The step is bound by HBM: every state byte is read once and written once
// and the arithmetic is 4 flops per state element.  One CTA owns one
// (batch, kv-head) state of Dk x Dv float32 (64 KiB at 128 x 128).  Warp w
// owns rows w, w+8, ..., lane c owns the four columns 4c..4c+3, so a warp
// moves one 512-byte row per 128-bit access (fully coalesced), and each
// thread keeps its 16 rows in registers between the load and the store so
// that all 16 loads are in flight at once.  Streaming cache hints keep the
// state, which is touched once per step, from displacing other data in L2.
// The read-out for every query head of the group is reduced across the
// eight warps in shared memory.
#include "common.cuh"
#include "kernels.h"

namespace la {

namespace {

constexpr int kThreads = 256;
constexpr int kRows = 16;     // rows per thread: Dk <= 128
constexpr int kHeadBlock = 4; // query heads reduced per round

struct DecArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* decay;
    float* S;
    float* Z;
    void* y;
    Problem P;
};

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(kThreads) decode_kernel(DecArgs a) {
    const Problem& P = a.P;
    const int Dk = P.Dk, Dv = P.Dv, G = P.G;
    extern __shared__ float smem[];
    float* fk = smem;                  // [128]
    float* vv = fk + 128;              // [128]
    float* zs = vv + 128;              // [128] updated Z
    float* den = zs + 128;             // [128]
    float* fq = den + 128;             // [G*Dk]
    float4* red = reinterpret_cast<float4*>(fq + ((G * Dk + 3) & ~3));  // [kHeadBlock][8][32]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t bh = blockIdx.x;
    const int64_t b = bh / P.Hkv;
    const int hk = (int)(bh % P.Hkv);
    const TIn* q = static_cast<const TIn*>(a.q);
    const TIn* k = static_cast<const TIn*>(a.k);
    const TIn* v = static_cast<const TIn*>(a.v);
    TOut* y = static_cast<TOut*>(a.y);
    const int nvec = Dv >> 2;  // float4 columns
    const bool colok = lane < nvec;

    // issue the state loads first: they are the long pole
    float4* Srow = reinterpret_cast<float4*>(a.S + bh * (int64_t)Dk * Dv);
    float4 s[kRows];
#pragma unroll
    for (int m = 0; m < kRows; ++m) {
        const int i = warp + 8 * m;
        s[m] = (i < Dk && colok) ? __ldcs(Srow + (int64_t)i * nvec + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
    }

    for (int i = tid; i < Dk; i += kThreads) fk[i] = phi<true>(P.fmap, load_in(k, bh * Dk + i), P.eps);
    for (int j = tid; j < Dv; j += kThreads) vv[j] = load_in(v, bh * Dv + j);
    for (int idx = tid; idx < G * Dk; idx += kThreads) {
        const int r = idx / Dk, i = idx - r * Dk;
        fq[idx] = phi<true>(P.fmap, load_in(q, (b * P.Hq + hk * G + r) * Dk + i), P.eps);
    }
    __syncthreads();
    if (P.norm && tid < Dk) {
        const float z = a.Z[bh * Dk + tid] + fk[tid];
        zs[tid] = z;
        a.Z[bh * Dk + tid] = z;
    }
    const float dec = P.gated ? __expf(load_in(static_cast<const TIn*>(a.decay), bh)) : 1.f;

    // S <- dec * S + phi(k) (x) v, written back in place
    const float4 v4 = colok ? reinterpret_cast<const float4*>(vv)[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < kRows; ++m) {
        const int i = warp + 8 * m;
        const float f = i < Dk ? fk[i] : 0.f;
        s[m].x = fmaf(f, v4.x, dec * s[m].x);
        s[m].y = fmaf(f, v4.y, dec * s[m].y);
        s[m].z = fmaf(f, v4.z, dec * s[m].z);
        s[m].w = fmaf(f, v4.w, dec * s[m].w);
        if (i < Dk && colok) __stcs(Srow + (int64_t)i * nvec + lane, s[m]);
    }
    __syncthreads();  // zs complete

    if (P.norm)
        for (int r = warp; r < G; r += 8) {
            float d = 0.f;
            for (int i = lane; i < Dk; i += 32) d = fmaf(fq[r * Dk + i], zs[i], d);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
            if (lane == 0) den[r] = d + P.eps;
        }
    for (int r0 = 0; r0 < G; r0 += kHeadBlock) {
        const int nh = min(kHeadBlock, G - r0);
        for (int rr = 0; rr < nh; ++rr) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int m = 0; m < kRows; ++m) {
                const int i = warp + 8 * m;
                const float f = i < Dk ? fq[(r0 + rr) * Dk + i] : 0.f;
                acc.x = fmaf(f, s[m].x, acc.x);
                acc.y = fmaf(f, s[m].y, acc.y);
                acc.z = fmaf(f, s[m].z, acc.z);
                acc.w = fmaf(f, s[m].w, acc.w);
            }
            red[(rr * 8 + warp) * 32 + lane] = acc;
        }
        __syncthreads();
        for (int idx = tid; idx < nh * Dv; idx += kThreads) {
            const int rr = idx / Dv, j = idx - rr * Dv;
            const float* rf = reinterpret_cast<const float*>(red);
            float num = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) num += rf[((rr * 8 + w) * 32) * 4 + j];
            const float out = P.norm ? num / den[r0 + rr] : num;
            store_out(y, (b * P.Hq + hk * G + r0 + rr) * Dv + j, P.scale * out);
        }
        __syncthreads();
    }
}

template <typename TIn, typename TOut>
cudaError_t launch(const DecArgs& a, cudaStream_t st) {
    const Problem& P = a.P;
    const size_t smem = sizeof(float) * (5 * 128 + (((size_t)P.G * P.Dk + 3) & ~(size_t)3)) +
                        sizeof(float4) * kHeadBlock * 8 * 32;
    auto kern = decode_kernel<TIn, TOut>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)(P.B * P.Hkv)), kThreads, smem, st>>>(a);
    note_launch();
    return cudaGetLastError();
}

}  // namespace

bool decode_supported(const Problem& P) { return P.Dk <= 128 && P.Dv <= 128 && P.Dv % 4 == 0; }

cudaError_t decode_step(const Problem& P, const void* q, const void* k, const void* v,
                        const void* decay, float* S, float* Z, void* y, cudaStream_t st) {
    DecArgs a{q, k, v, decay, S, Z, y, P};
    if (P.io_bf16)
        return P.out_bf16 ? launch<__nv_bfloat16, __nv_bfloat16>(a, st) : launch<__nv_bfloat16, float>(a, st);
    return P.out_bf16 ? launch<float, __nv_bfloat16>(a, st) : launch<float, float>(a, st);
}

}  // namespace la
