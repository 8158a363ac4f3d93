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
//
// A sequence-validity mask (Keras request, Masking) makes a sequence's step
// invalid: its state and key sum are left exactly as they were and its
// outputs are zero.  The decision is per batch row, uniform across a CTA.
// The mask and the per-key-dimension decay are compiled into separate
// instantiations (EXT); the plain step carries no code for either.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "umma.cuh"

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

template <typename TIn, typename TOut, bool EXT>
__global__ void __launch_bounds__(kThreads) decode_kernel(DecArgs a) {
    const Problem& P = a.P;
    const uint8_t* mask = EXT ? P.mask : nullptr;     // sequence-validity mask
    const bool decay_dim = EXT && P.gated && P.decay_dim;  // decay per key dimension
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
    const bool valid = step_valid(mask, b);
    if (!valid) {  // state untouched, zero outputs
        for (int idx = tid; idx < G * Dv; idx += kThreads) store_out(y, (b * P.Hq + hk * G) * Dv + idx, 0.f);
        return;
    }
    if (P.norm && tid < Dk) {
        const float z = a.Z[bh * Dk + tid] + fk[tid];
        zs[tid] = z;
        a.Z[bh * Dk + tid] = z;
    }
    const TIn* dg = static_cast<const TIn*>(a.decay);
    const float dec = P.gated && !decay_dim ? __expf(load_in(dg, bh)) : 1.f;

    // S <- dec * S + phi(k) (x) v, written back in place (per-key-dimension
    // decay: row i scaled by its own exp(g_i))
    const float4 v4 = colok ? reinterpret_cast<const float4*>(vv)[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < kRows; ++m) {
        const int i = warp + 8 * m;
        const float f = i < Dk ? fk[i] : 0.f;
        const float di = decay_dim && i < Dk ? __expf(load_in(dg, bh * Dk + i)) : dec;
        s[m].x = fmaf(f, v4.x, di * s[m].x);
        s[m].y = fmaf(f, v4.y, di * s[m].y);
        s[m].z = fmaf(f, v4.z, di * s[m].z);
        s[m].w = fmaf(f, v4.w, di * s[m].w);
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

// ------------------------------------------------------------ streamed decode
// The same step as decode_kernel, organised for bandwidth: a persistent CTA per
// SM walks the (batch, kv head) units blockIdx.x, + gridDim.x, ... and streams
// each unit's state through a ring of shared-memory stages with bulk async
// copies (TMA): the loads of the next units are in flight while a unit is
// updated, and the updated state drains back with a bulk store while the
// read-out runs.  The unit's k, v, q and key sum come with its state.
struct StreamLayout {
    int S, k, v, q, z;  // byte offsets inside a stage
    int stage;          // stage size (multiple of 128)
    int nst;            // stages (2 or 3)
    int smem;           // dynamic shared memory of the kernel
};

using namespace umma;

template <typename TIn, typename TOut, bool EXT>
__global__ void __launch_bounds__(kThreads, 1)
    decode_stream_kernel(DecArgs a, StreamLayout ly, int nunits, unsigned* err) {
    const Problem& P = a.P;
    const uint8_t* mask = EXT ? P.mask : nullptr;     // sequence-validity mask
    const bool decay_dim = EXT && P.gated && P.decay_dim;  // decay per key dimension
    const int Dk = P.Dk, Dv = P.Dv, G = P.G, nst = ly.nst;
    extern __shared__ __align__(128) uint8_t dsm[];
    uint8_t* stages = dsm;
    float4* red = reinterpret_cast<float4*>(dsm + nst * ly.stage);  // [kHeadBlock][8][32]
    float* fk = reinterpret_cast<float*>(red + kHeadBlock * 8 * 32);  // [128]
    float* vv = fk + 128;
    float* zs = vv + 128;
    float* den = zs + 128;
    float* fq = den + 128;  // [G*Dk]
    uint64_t* full = reinterpret_cast<uint64_t*>(fq + ((G * Dk + 1) & ~1));  // [nst]
    int* flag = reinterpret_cast<int*>(full + 3);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nvec = Dv >> 2;
    const bool colok = lane < nvec;
    const int esz = sizeof(TIn);
    const TIn* q = static_cast<const TIn*>(a.q);
    const TIn* k = static_cast<const TIn*>(a.k);
    const TIn* v = static_cast<const TIn*>(a.v);
    TOut* y = static_cast<TOut*>(a.y);
    const uint32_t sbytes = (uint32_t)Dk * Dv * 4;

    // the units of this CTA: j = 0, 1, ... -> u = blockIdx.x + j * gridDim.x
    const int nj = blockIdx.x < nunits ? (nunits - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    auto issue_load = [&](int j) {  // thread 0
        const int64_t u = blockIdx.x + (int64_t)j * gridDim.x;
        const int64_t b = u / P.Hkv, hk = u - b * P.Hkv;
        uint8_t* st = stages + (j % nst) * ly.stage;
        const uint32_t qb = (uint32_t)(G * Dk * esz), kb = (uint32_t)(Dk * esz), vb = (uint32_t)(Dv * esz);
        const uint32_t zb = P.norm ? (uint32_t)Dk * 4 : 0;
        mbar_arrive_expect_tx(&full[j % nst], sbytes + kb + vb + qb + zb);
        bulk_load(st + ly.S, a.S + u * Dk * Dv, sbytes, &full[j % nst]);
        bulk_load(st + ly.k, k + u * Dk, kb, &full[j % nst]);
        bulk_load(st + ly.v, v + u * Dv, vb, &full[j % nst]);
        bulk_load(st + ly.q, q + (b * P.Hq + hk * G) * Dk, qb, &full[j % nst]);
        if (P.norm) bulk_load(st + ly.z, a.Z + u * Dk, zb, &full[j % nst]);
    };
    if (tid == 0) {
        for (int i = 0; i < nst; ++i) mbar_init(&full[i], 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0)
        for (int j = 0; j < nst - 1 && j < nj; ++j) issue_load(j);

    for (int j = 0; j < nj; ++j) {
        const int64_t u = blockIdx.x + (int64_t)j * gridDim.x;
        const int64_t b = u / P.Hkv;
        const int hk = (int)(u - b * P.Hkv);
        uint8_t* st = stages + (j % nst) * ly.stage;
        // the stage has landed: a bounded wait by one thread, its outcome shared
        if (tid == 0) *flag = mbar_wait(&full[j % nst], (j / nst) & 1, err, 1u << 16);
        __syncthreads();
        if (!*flag) break;
        mbar_try_wait(&full[j % nst], (j / nst) & 1);  // acquire for this thread as well

        float4* Ss = reinterpret_cast<float4*>(st + ly.S);
        float4 s[kRows];
#pragma unroll
        for (int m = 0; m < kRows; ++m) {
            const int i = warp + 8 * m;
            s[m] = (i < Dk && colok) ? Ss[i * nvec + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        const TIn* ks = reinterpret_cast<const TIn*>(st + ly.k);
        const TIn* vs = reinterpret_cast<const TIn*>(st + ly.v);
        const TIn* qs = reinterpret_cast<const TIn*>(st + ly.q);
        for (int i = tid; i < Dk; i += kThreads) fk[i] = phi<true>(P.fmap, load_in(ks, i), P.eps);
        for (int jv = tid; jv < Dv; jv += kThreads) vv[jv] = load_in(vs, jv);
        for (int idx = tid; idx < G * Dk; idx += kThreads) fq[idx] = phi<true>(P.fmap, load_in(qs, idx), P.eps);
        __syncthreads();
        // an invalid step (mask) keeps the stage as loaded: the store below
        // then writes the state back unchanged
        const bool valid = step_valid(mask, b);
        if (valid && P.norm && tid < Dk) {
            const float z = reinterpret_cast<const float*>(st + ly.z)[tid] + fk[tid];
            zs[tid] = z;
            a.Z[u * Dk + tid] = z;
        }
        const TIn* dg = static_cast<const TIn*>(a.decay);
        const float dec = P.gated && !decay_dim ? __expf(load_in(dg, u)) : 1.f;
        // S <- dec * S + phi(k) (x) v, written back into the stage (row i
        // scaled by its own exp(g_i) with the per-key-dimension decay)
        const float4 v4 = colok ? reinterpret_cast<const float4*>(vv)[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
        if (valid) {
#pragma unroll
            for (int m = 0; m < kRows; ++m) {
                const int i = warp + 8 * m;
                const float f = i < Dk ? fk[i] : 0.f;
                const float di = decay_dim && i < Dk ? __expf(load_in(dg, u * Dk + i)) : dec;
                s[m].x = fmaf(f, v4.x, di * s[m].x);
                s[m].y = fmaf(f, v4.y, di * s[m].y);
                s[m].z = fmaf(f, v4.z, di * s[m].z);
                s[m].w = fmaf(f, v4.w, di * s[m].w);
                if (i < Dk && colok) Ss[i * nvec + lane] = s[m];
            }
        }
        fence_proxy_async();  // this thread's state writes, before the bulk store reads them
        __syncthreads();      // every state row written; zs complete
        if (tid == 0) {
            bulk_store(a.S + u * Dk * Dv, st + ly.S, sbytes);
            bulk_commit_group();
            // the stage of unit j - 1 is read out by its store: refill it
            bulk_wait_group_read<1>();
            if (j + nst - 1 < nj) issue_load(j + nst - 1);
        }
        if (!valid) {  // uniform across the CTA
            for (int idx = tid; idx < G * Dv; idx += kThreads) store_out(y, (b * P.Hq + hk * G) * Dv + idx, 0.f);
            continue;
        }

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
                const int rr = idx / Dv, jv = idx - rr * Dv;
                const float* rf = reinterpret_cast<const float*>(red);
                float num = 0.f;
#pragma unroll
                for (int w = 0; w < 8; ++w) num += rf[((rr * 8 + w) * 32) * 4 + jv];
                const float out = P.norm ? num / den[r0 + rr] : num;
                store_out(y, (b * P.Hq + hk * G + r0 + rr) * Dv + jv, P.scale * out);
            }
            __syncthreads();
        }
    }
    // the stores must finish reading shared memory before the CTA exits
    if (tid == 0) bulk_wait_group<0>();
}

template <typename TIn, typename TOut, bool EXT>
cudaError_t launch(const DecArgs& a, cudaStream_t st) {
    const Problem& P = a.P;
    const size_t smem = sizeof(float) * (5 * 128 + (((size_t)P.G * P.Dk + 3) & ~(size_t)3)) +
                        sizeof(float4) * kHeadBlock * 8 * 32;
    auto kern = decode_kernel<TIn, TOut, EXT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)(P.B * P.Hkv)), kThreads, smem, st>>>(a);
    note_launch();
    return cudaGetLastError();
}

// Stage layout of the streamed kernel, or nst = 0 when it does not apply: the
// bulk copies need 16-byte aligned addresses and sizes, and at least two
// stages must fit in shared memory.
StreamLayout stream_layout(const Problem& P, const void* q, const void* k, const void* v, const float* S,
                           const float* Z) {
    StreamLayout ly{};
    const int esz = P.io_bf16 ? 2 : 4;
    auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    auto up = [](int x, int m) { return (x + m - 1) / m * m; };
    if ((P.Dk * esz) % 16 || (P.Dv * esz) % 16 || P.Dv % 4 || !al16(q) || !al16(k) || !al16(v) || !al16(S) ||
        (P.norm && !al16(Z)))
        return ly;
    ly.S = 0;
    ly.k = P.Dk * P.Dv * 4;
    ly.v = ly.k + up(P.Dk * esz, 16);
    ly.q = ly.v + up(P.Dv * esz, 16);
    ly.z = ly.q + up(P.G * P.Dk * esz, 16);
    ly.stage = up(ly.z + P.Dk * 4, 128);
    const int fixed = kHeadBlock * 8 * 32 * 16 + 4 * 128 * 4 + ((P.G * P.Dk + 1) & ~1) * 4 + 4 * 8;
    for (int nst = 3; nst >= 2; --nst)
        if (nst * ly.stage + fixed <= 227 * 1024) {
            ly.nst = nst;
            ly.smem = nst * ly.stage + fixed;
            return ly;
        }
    ly.nst = 0;
    return ly;
}

template <typename TIn, typename TOut, bool EXT>
cudaError_t launch_stream(const DecArgs& a, const StreamLayout& ly, cudaStream_t st) {
    const int nunits = (int)(a.P.B * a.P.Hkv);
    const int sms = device_sm_count();
    unsigned* err = device_error_word();
    if (sms <= 0 || !err) return cudaErrorInvalidDevice;
    auto kern = decode_stream_kernel<TIn, TOut, EXT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, ly.smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)std::min(nunits, sms)), kThreads, ly.smem, st>>>(a, ly, nunits, err);
    note_launch();
    return cudaGetLastError();
}

}  // namespace

bool decode_supported(const Problem& P) { return P.Dk <= 128 && P.Dv <= 128 && P.Dv % 4 == 0; }

template <bool EXT>
cudaError_t decode_dispatch(const DecArgs& a, const StreamLayout& ly, cudaStream_t st) {
    const Problem& P = a.P;
    if (ly.nst) {  // state streamed through shared memory (bulk async copies)
        if (P.io_bf16)
            return P.out_bf16 ? launch_stream<__nv_bfloat16, __nv_bfloat16, EXT>(a, ly, st)
                              : launch_stream<__nv_bfloat16, float, EXT>(a, ly, st);
        return P.out_bf16 ? launch_stream<float, __nv_bfloat16, EXT>(a, ly, st)
                          : launch_stream<float, float, EXT>(a, ly, st);
    }
    if (P.io_bf16)
        return P.out_bf16 ? launch<__nv_bfloat16, __nv_bfloat16, EXT>(a, st) : launch<__nv_bfloat16, float, EXT>(a, st);
    return P.out_bf16 ? launch<float, __nv_bfloat16, EXT>(a, st) : launch<float, float, EXT>(a, st);
}

cudaError_t decode_step(const Problem& P, const void* q, const void* k, const void* v,
                        const void* decay, float* S, float* Z, void* y, cudaStream_t st) {
    DecArgs a{q, k, v, decay, S, Z, y, P};
    const StreamLayout ly = stream_layout(P, q, k, v, S, Z);
    // a mask or a per-key-dimension decay: the instantiations that read them
    if (P.mask || (P.gated && P.decay_dim)) return decode_dispatch<true>(a, ly, st);
    return decode_dispatch<false>(a, ly, st);
}

}  // namespace la
