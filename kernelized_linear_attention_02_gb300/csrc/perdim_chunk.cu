// perdim_chunk.cu -- the gated rule with one log decay per key dimension
// (ONNX-light "LinearAttention", decay of shape (B, T, H_kv * d_k), as in
// GLA / RWKV-6) in chunk-parallel form on the tensor cores, for bf16 inputs
// with Dk = Dv = 128.
//
// Per (batch, kv head) stream and chunk of C = 64 steps with start state S0,
// G_t[k] the inclusive cumulative log decay of key dimension k inside the
// chunk (a step that is masked out or past T has g = 0 and zero key and value
// rows):
//   S_t = diag(e^{g_t}) S_{t-1} + k_t v_t^T
//   =>  S_C = diag(e^{G_C}) S0 + Khat^T V,   Khat[l][k] = k_l[k] e^{G_C[k] - G_l[k]}
//       o_t = S0^T (q_t o e^{G_t}) + sum_{l<=t} v_l sum_k q_t[k] k_l[k] e^{G_t[k] - G_l[k]}
// The intra weights factor per key dimension: with Qbar = q o e^{G} and
// Kbar = k o e^{-G} the scores are Qbar Kbar^T, exact as long as every
// factor stays in float32 range; a chunk whose cumulative decay leaves
// (-kFactorRange, kFactorRange) in some dimension (log decays below about
// -1.25 per step on average) computes its intra scores on CUDA cores with one
// exponential per term instead.
//
// Three kernels, in stream order: prep (one CTA per chunk: Khat and
// N = Khat^T V on the tensor cores, and the chunk's transition diag(e^{G_C})
// as a vector), scan (S_{c+1} = diag(e^{G_C}) S_c + N_c element by element:
// the transition is diagonal, so each state element is its own scalar
// recurrence and the scan spreads over every element of every stream), and
// out (one CTA per chunk: the outputs of every query head).  Every fp32
// operand enters the tensor cores as bf16 hi + lo; keys, values and queries
// that enter unscaled are exact.
#include <algorithm>
#include <atomic>
#include <cstring>

#include "delta_args.h"
#include "kernels.h"
#include "tiles.cuh"
#include "umma.cuh"

namespace la {
namespace perdim {

using namespace umma;
using namespace tile;
using delta::Args;
using delta::Ws;

constexpr int kC = 64;
constexpr int kD = 128;
constexpr float kMinLogDecay = -200.f;  // a -inf step: exp of it is zero in float32
constexpr float kFactorRange = 80.f;    // |G| below this keeps e^{+-G} (times a bounded input) in range

enum : unsigned { kErrLoad = 1u << 18, kErrMma = 1u << 19 };

// Validity of the chunk's 64 steps as a word (bit t: step t0 + t is inside T
// and not masked out); warp-collective.
__device__ __forceinline__ uint64_t valid_word(const Args& a, int b, int t0) {
    const int lane = threadIdx.x & 31;
    auto valid = [&](int j) {
        const int t = t0 + j;
        return t < a.T && (!a.mask || a.mask[(size_t)b * a.T + t] != 0);
    };
    return step_word(valid(2 * lane), valid(2 * lane + 1));
}

// eight consecutive floats of shared memory (32-byte aligned) in two 16-byte loads
__device__ __forceinline__ void load_g8(const float* p, float (&g)[8]) {
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    g[0] = a.x, g[1] = a.y, g[2] = a.z, g[3] = a.w, g[4] = b.x, g[5] = b.y, g[6] = b.z, g[7] = b.w;
}

// The log decays of a chunk's steps, loaded as 16-byte chunks (chunk i of
// thread `th`: step e / 16, key dimensions 8 (e % 16) .. + 7, e = th + nthr i;
// zero for masked-out steps and steps past T), floored at kMinLogDecay into G[t][k].
template <int kN>
__device__ __forceinline__ void store_decays(float* Gs, const uint4 (&dq)[kN], int th, int nthr) {
#pragma unroll
    for (int i = 0; i < kN; ++i) {
        const int e = th + nthr * i, l = e >> 4, k0 = 8 * (e & 15);
        const __nv_bfloat16* p = reinterpret_cast<const __nv_bfloat16*>(&dq[i]);
        float g[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) g[x] = fmaxf(__bfloat162float(p[x]), kMinLogDecay);
        *reinterpret_cast<float4*>(Gs + l * kD + k0) = make_float4(g[0], g[1], g[2], g[3]);
        *reinterpret_cast<float4*>(Gs + l * kD + k0 + 4) = make_float4(g[4], g[5], g[6], g[7]);
    }
}

// ------------------------------------------------------------------ prep
struct PrepSmem {
    static constexpr int kKh = 0;       // Khat, rows l (64), k in 2 blocks of 8 KB: hi 16 KB, lo 16 KB
    static constexpr int kV = 32768;    // V, rows l, v in 2 blocks of 8 KB
    static constexpr int kG = 49152;    // G fp32 [64][128]
    static constexpr int kW = kG + 32768;  // validity word
    static constexpr int kBar = kW + 64;
    static constexpr int kBytes = kBar + 64 + 1024;
};

__global__ void __launch_bounds__(128, 1)
    perdim_prep_kernel(const __grid_constant__ Args a, const __nv_bfloat16* __restrict__ kin,
                       const __nv_bfloat16* __restrict__ vin) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* Kh = sm + PrepSmem::kKh;
    uint8_t* Vt = sm + PrepSmem::kV;
    uint64_t* s_word = reinterpret_cast<uint64_t*>(sm + PrepSmem::kW);
    uint64_t* bar_mma = reinterpret_cast<uint64_t*>(sm + PrepSmem::kBar);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bar_mma + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x / a.nc, c = blockIdx.x - bh * a.nc;
    const int b = bh / a.Hkv, hk = bh - b * a.Hkv;
    const int t0 = c * kC;
    uint8_t* wsc = a.ws + ((size_t)bh * a.nc + c) * Ws::kChunk;

    if (tid == 0) {
        mbar_init(bar_mma, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        const uint64_t w = valid_word(a, b, t0);
        if (lane == 0) *s_word = w;
        tmem_alloc(tslot, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint64_t vw = *s_word;

    {
        // the chunk's keys and values as 16-byte chunks (row l, eight key or
        // value dimensions), all in flight while the decays load and sum
        constexpr int kIt = kC * (kD / 8) / 128;
        uint4 kq[kIt], vq[kIt], dq[kIt];
#pragma unroll
        for (int i = 0; i < kIt; ++i) {
            const int e = tid + 128 * i, l = e >> 4, cc = e & 15;
            const size_t row = ((size_t)b * a.T + t0 + l) * a.Hkv + hk;
            const bool ok = (vw >> l) & 1;
            kq[i] = ok ? *reinterpret_cast<const uint4*>(kin + row * kD + 8 * cc) : make_uint4(0, 0, 0, 0);
            vq[i] = ok ? *reinterpret_cast<const uint4*>(vin + row * kD + 8 * cc) : make_uint4(0, 0, 0, 0);
            dq[i] = ok ? *reinterpret_cast<const uint4*>(a.decay + row * kD + 8 * cc) : make_uint4(0, 0, 0, 0);
        }
        float* Gs = reinterpret_cast<float*>(sm + PrepSmem::kG);
        store_decays(Gs, dq, tid, 128);
        __syncthreads();
        // key dimension k = tid: cumulative decay down the chunk, in place
        const int k = tid;
        float G = 0.f;
#pragma unroll 8
        for (int t = 0; t < kC; ++t) {
            G += Gs[t * kD + k];
            Gs[t * kD + k] = G;
        }
        // the chunk's transition is diagonal: gamma[k] = e^{G_C[k]}, fp32
        reinterpret_cast<float*>(wsc + Ws::kG)[k] = __expf(G);
        __syncthreads();  // every column of G (G_C in its last row)
        // Khat[l][k] = k_l[k] e^{G_C[k] - G_l[k]} (hi, lo) and V into the (rows l) tiles
#pragma unroll
        for (int i = 0; i < kIt; ++i) {
            const int e = tid + 128 * i, l = e >> 4, cc = e & 15, k0 = 8 * cc;
            float f[8], gl[8], gc[8];
            const __nv_bfloat16* kp = reinterpret_cast<const __nv_bfloat16*>(&kq[i]);
#pragma unroll
            for (int x = 0; x < 8; ++x) f[x] = __bfloat162float(kp[x]);
            load_g8(Gs + l * kD + k0, gl);
            load_g8(Gs + (kC - 1) * kD + k0, gc);
#pragma unroll
            for (int x = 0; x < 8; ++x) f[x] *= __expf(gc[x] - gl[x]);
            uint4 hi, lo;
            split8(f, hi, lo);
            const uint32_t off = (cc >> 3) * 8192 + swc(l, cc & 7);
            st16(Kh + off, hi);
            st16(Kh + 16384 + off, lo);
            st16(Vt + off, vq[i]);  // values exact
        }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        tc_fence_after();
        // N^T[v][k] = sum_l V[l][v] Khat[l][k]: A = V (rows l, M = v), B = Khat (rows l, N = k)
        constexpr uint32_t id = idesc_bf16(128, 128, true, true);
#pragma unroll 1
        for (int ks = 0; ks < kC / 16; ++ks) {
            const uint64_t av = sdesc_sw128(smem_u32(Vt + ks * 2048), 8192, 1024);
            mma_ss(tmem, av, sdesc_sw128(smem_u32(Kh + ks * 2048), 8192, 1024), id, ks > 0);
            mma_ss(tmem, av, sdesc_sw128(smem_u32(Kh + 16384 + ks * 2048), 8192, 1024), id, 1);
        }
        mma_commit(bar_mma);
    }
    warp_wait(bar_mma, 0, a.err, kErrMma);
    tc_fence_after();
    {
        float* nt = reinterpret_cast<float*>(wsc + Ws::kN);
        const int v = tid;
#pragma unroll 1
        for (int p = 0; p < 4; ++p) {
            uint32_t r[32];
            tmem_ld32(tmem_addr(tmem, warp * 32, 32 * p), r);
            tmem_ld_wait();
            reg_fence(r);
#pragma unroll
            for (int x = 0; x < 32; ++x) nt[(32 * p + x) * kD + v] = __uint_as_float(r[x]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}

// ------------------------------------------------------------------ scan
// Thread (v, kg) of a stream carries S[8 kg .. 8 kg + 7][v] in fp32 through the
// chunks.  Per chunk it writes the start state into the chunk's S^T tile (row
// v, the 16-byte group of keys 8 kg .. 8 kg + 7, hi and lo), then applies
// S <- gamma o S + N.  Loads run kScanDepth chunks ahead of the recurrence.
constexpr int kScanThreads = 256;  // 32 values x 8 key groups
constexpr int kScanCtas = 8;       // per stream: 4 value blocks x 2 key-group halves
constexpr int kScanDepth = 8;

__global__ void __launch_bounds__(kScanThreads) perdim_scan_kernel(const __grid_constant__ Args a) {
    const int bh = blockIdx.x / kScanCtas, j = blockIdx.x - bh * kScanCtas;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int v = 32 * (j & 3) + lane, k0 = 8 * (8 * (j >> 2) + warp);
    const int nc = a.nc;
    uint8_t* ws0 = a.ws + (size_t)bh * nc * Ws::kChunk;
    const uint32_t soff = (k0 >> 6) * 16384 + swc(v, (k0 & 63) >> 3);

    float S[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) S[i] = a.S0 ? a.S0[(size_t)bh * kD * kD + (size_t)(k0 + i) * kD + v] : 0.f;

    float nb[kScanDepth][8], gb[kScanDepth][8];
    auto load = [&](int c, float (&n)[8], float (&g)[8]) {
        const uint8_t* w = ws0 + (size_t)c * Ws::kChunk;
        const float* nt = reinterpret_cast<const float*>(w + Ws::kN);
#pragma unroll
        for (int i = 0; i < 8; ++i) n[i] = nt[(k0 + i) * kD + v];
        const float4 g0 = *reinterpret_cast<const float4*>(w + Ws::kG + 4 * k0);
        const float4 g1 = *reinterpret_cast<const float4*>(w + Ws::kG + 4 * k0 + 16);
        g[0] = g0.x, g[1] = g0.y, g[2] = g0.z, g[3] = g0.w;
        g[4] = g1.x, g[5] = g1.y, g[6] = g1.z, g[7] = g1.w;
    };
#pragma unroll
    for (int i = 0; i < kScanDepth; ++i)
        if (i < nc) load(i, nb[i], gb[i]);
#pragma unroll 1
    for (int c0 = 0; c0 < nc; c0 += kScanDepth) {
#pragma unroll
        for (int i = 0; i < kScanDepth; ++i) {
            const int c = c0 + i;
            if (c < nc) {
                uint4 hi, lo;
                split8(S, hi, lo);
                uint8_t* st = ws0 + (size_t)c * Ws::kChunk + Ws::kS;
                st16(st + soff, hi);
                st16(st + 32768 + soff, lo);
#pragma unroll
                for (int x = 0; x < 8; ++x) S[x] = fmaf(gb[i][x], S[x], nb[i][x]);
                if (c + kScanDepth < nc) load(c + kScanDepth, nb[i], gb[i]);
            }
        }
    }
    if (a.S_out) {
#pragma unroll
        for (int i = 0; i < 8; ++i) a.S_out[(size_t)bh * kD * kD + (size_t)(k0 + i) * kD + v] = S[i];
    }
}

// ------------------------------------------------------------------ out
struct OutSmem {
    static constexpr int kKb = 0;        // Kbar as B operand (rows l, K = k, 2 blocks of 8 KB): hi, lo
    static constexpr int kV = 32768;     // V as A operand (rows l, v contiguous), 2 blocks of 8 KB
    static constexpr int kQ = 49152;     // Qbar of a head pair (rows (r, t), K = k, 2 blocks of 16 KB): hi, lo
    static constexpr int kP = 114688;    // P (rows (r, t), K = l): hi, lo (16 KB each)
    static constexpr int kG = 147456;    // G fp32 [64][128]
    static constexpr int kW = kG + 32768;
    static constexpr int kBar = kW + 64;
    static constexpr int kBytes = kBar + 64 + 1024;
};
constexpr uint32_t kOutSHi = 0, kOutSLo = 64, kOutX = 128, kOutSP = 256, kOutY = 384;

__global__ void __launch_bounds__(256, 1)
    perdim_out_kernel(const __grid_constant__ Args a, const __nv_bfloat16* __restrict__ q,
                      const __nv_bfloat16* __restrict__ kin, const __nv_bfloat16* __restrict__ vin) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* Kb = sm + OutSmem::kKb;
    uint8_t* Vt = sm + OutSmem::kV;
    uint8_t* Qb = sm + OutSmem::kQ;
    uint8_t* Pp = sm + OutSmem::kP;
    float* Gs = reinterpret_cast<float*>(sm + OutSmem::kG);
    uint64_t* s_word = reinterpret_cast<uint64_t*>(sm + OutSmem::kW);
    uint64_t* bar_mma = reinterpret_cast<uint64_t*>(sm + OutSmem::kBar);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bar_mma + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3;
    const int bh = blockIdx.x / a.nc, c = blockIdx.x - bh * a.nc;
    const int b = bh / a.Hkv, hk = bh - b * a.Hkv;
    const int t0 = c * kC, G = a.G;
    const uint8_t* wsc = a.ws + ((size_t)bh * a.nc + c) * Ws::kChunk;
    unsigned* err = a.err;

    if (tid == 0) {
        mbar_init(bar_mma, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        const uint64_t w = valid_word(a, b, t0);
        if (lane == 0) *s_word = w;
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint64_t vw = *s_word;
    bool fac = true;
    if (warp < 4) {
        // the chunk's start state: row v of S^T (hi, lo) from the scan's tile into TMEM
        const int v = quad * 32 + lane;
        const uint8_t* st = wsc + Ws::kS;
#pragma unroll 1
        for (int p0 = 0; p0 < 4; p0 += 2) {
            // two 32-key blocks (hi and lo) in flight, then their four TMEM stores
            uint32_t h[2][16], l[2][16];
#pragma unroll
            for (int pp = 0; pp < 2; ++pp)
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int k0 = 32 * (p0 + pp) + 8 * q4;
                    const uint32_t off = (k0 >> 6) * 16384 + swc(v, (k0 & 63) >> 3);
                    const uint4 hh = *reinterpret_cast<const uint4*>(st + off);
                    const uint4 ll = *reinterpret_cast<const uint4*>(st + 32768 + off);
                    h[pp][4 * q4] = hh.x, h[pp][4 * q4 + 1] = hh.y, h[pp][4 * q4 + 2] = hh.z, h[pp][4 * q4 + 3] = hh.w;
                    l[pp][4 * q4] = ll.x, l[pp][4 * q4 + 1] = ll.y, l[pp][4 * q4 + 2] = ll.z, l[pp][4 * q4 + 3] = ll.w;
                }
#pragma unroll
            for (int pp = 0; pp < 2; ++pp) {
                tmem_st16(tmem_addr(tmem + kOutSHi, quad * 32, 16 * (p0 + pp)), h[pp]);
                tmem_st16(tmem_addr(tmem + kOutSLo, quad * 32, 16 * (p0 + pp)), l[pp]);
            }
        }
        tmem_st_wait();
    } else {
        // the chunk's log decays into G (warps 4-7), then the cumulative decay
        // of key dimension k down the chunk, in place
        const int k = tid - 128;
        uint4 dq[kC * (kD / 8) / 128];
#pragma unroll
        for (int i = 0; i < kC * (kD / 8) / 128; ++i) {
            const int e = k + 128 * i, l = e >> 4, cc = e & 15;
            const size_t row = ((size_t)b * a.T + t0 + l) * a.Hkv + hk;
            dq[i] = ((vw >> l) & 1) ? *reinterpret_cast<const uint4*>(a.decay + row * kD + 8 * cc)
                                    : make_uint4(0, 0, 0, 0);
        }
        store_decays(Gs, dq, k, 128);
        named_bar_sync(1, 128);  // warps 4-7
        float G_ = 0.f, mn = 0.f, mx = 0.f;
#pragma unroll 8
        for (int t = 0; t < kC; ++t) {
            G_ += Gs[t * kD + k];
            Gs[t * kD + k] = G_;
            mn = fminf(mn, G_);
            mx = fmaxf(mx, G_);
        }
        fac = mn > -kFactorRange && mx < kFactorRange;
    }
    fac = __syncthreads_and(fac);  // G complete; the whole chunk factors (or not)

    // Kbar (only when the chunk factors) and V, rows l
#pragma unroll
    for (int e = tid; e < kC * 16; e += 256) {
        const int l = e >> 4, cc = e & 15, k0 = 8 * cc;
        const bool ok = (vw >> l) & 1;
        const size_t row = ((size_t)b * a.T + t0 + l) * a.Hkv + hk;
        const uint32_t off = (cc >> 3) * 8192 + swc(l, cc & 7);
        uint4 vv = make_uint4(0, 0, 0, 0), kk = make_uint4(0, 0, 0, 0);
        if (ok) {
            vv = *reinterpret_cast<const uint4*>(vin + row * kD + k0);
            kk = *reinterpret_cast<const uint4*>(kin + row * kD + k0);
        }
        *reinterpret_cast<uint4*>(Vt + off) = vv;
        if (fac) {
            float f[8], g8[8];
            load_g8(Gs + l * kD + k0, g8);
            const __nv_bfloat16* kp = reinterpret_cast<const __nv_bfloat16*>(&kk);
#pragma unroll
            for (int x = 0; x < 8; ++x) f[x] = __bfloat162float(kp[x]) * __expf(-g8[x]);
            uint4 hi, lo;
            split8(f, hi, lo);
            st16(Kb + off, hi);
            st16(Kb + 16384 + off, lo);
        }
    }

    constexpr uint32_t id128 = idesc_bf16(128, 128, false, false);
    constexpr uint32_t id64 = idesc_bf16(128, 64, false, false);
    constexpr uint32_t idy = idesc_bf16(128, 128, true, false);
    uint32_t mma_phase = 0;
    bool ok = true;
    const int npairs = (G + 1) / 2;
    // Qbar of query heads 2 pr and 2 pr + 1: rows (r, t), q o e^{G_t}, built by
    // nthr threads (the loads of eight rows in flight before their stores)
    auto build_qbar = [&](int pr, int bt, int nthr) {
#pragma unroll 1
        for (int e0 = bt; e0 < 128 * 16; e0 += 8 * nthr) {
            uint4 qq[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int e = e0 + u * nthr, row = e >> 4, cc = e & 15, r = row >> 6, t = row & 63;
                const int hq = 2 * pr + r;
                qq[u] = (e < 128 * 16 && hq < G && ((vw >> t) & 1))
                            ? *reinterpret_cast<const uint4*>(
                                  q + (((size_t)b * a.T + t0 + t) * a.Hq + (size_t)hk * G + hq) * kD + 8 * cc)
                            : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int e = e0 + u * nthr;
                if (e >= 128 * 16) continue;
                const int row = e >> 4, cc = e & 15, k0 = 8 * cc, t = row & 63;
                const __nv_bfloat16* qp = reinterpret_cast<const __nv_bfloat16*>(&qq[u]);
                float f[8], g8[8];
                load_g8(Gs + t * kD + k0, g8);
#pragma unroll
                for (int x = 0; x < 8; ++x) f[x] = __bfloat162float(qp[x]) * __expf(g8[x]);
                uint4 hi, lo;
                split8(f, hi, lo);
                const uint32_t off = (cc >> 3) * 16384 + swc(row, cc & 7);
                st16(Qb + off, hi);
                st16(Qb + 32768 + off, lo);
            }
        }
    };
    if (npairs > 0) build_qbar(0, tid, 256);
#pragma unroll 1
    for (int pr = 0; pr < npairs && ok; ++pr) {
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
#pragma unroll 1
            for (int ks = 0; ks < kD / 16; ++ks) {
                const uint32_t qo = (ks >> 2) * 16384 + (ks & 3) * 32;
                const uint64_t qh = sdesc_sw128(smem_u32(Qb + qo), 16, 1024);
                const uint64_t ql = sdesc_sw128(smem_u32(Qb + 32768 + qo), 16, 1024);
                // X = S^T Qbar^T (rows v, columns (r, t))
                mma_ts(tmem + kOutX, tmem + kOutSHi + ks * 8, qh, id128, ks > 0);
                mma_ts(tmem + kOutX, tmem + kOutSHi + ks * 8, ql, id128, 1);
                mma_ts(tmem + kOutX, tmem + kOutSLo + ks * 8, qh, id128, 1);
                if (fac) {
                    // scores Qbar Kbar^T (rows (r, t), columns l)
                    const uint32_t ko = (ks >> 2) * 8192 + (ks & 3) * 32;
                    const uint64_t kh = sdesc_sw128(smem_u32(Kb + ko), 16, 1024);
                    const uint64_t kl = sdesc_sw128(smem_u32(Kb + 16384 + ko), 16, 1024);
                    mma_ss(tmem + kOutSP, qh, kh, id64, ks > 0);
                    mma_ss(tmem + kOutSP, qh, kl, id64, 1);
                    mma_ss(tmem + kOutSP, ql, kh, id64, 1);
                }
            }
            mma_commit(bar_mma);
        }
        ok = warp_wait(bar_mma, mma_phase++ & 1, err, kErrMma);
        ok = __syncthreads_and(ok);
        if (!ok) break;
        tc_fence_after();
        // X and the scores have read this pair's Qbar: warps 0-3 build the next
        // pair's while warps 4-7 build P
        if (warp < 4 && pr + 1 < npairs) build_qbar(pr + 1, tid, 128);
        if (warp >= 4) {
            // P rows (r, t): masked scores, l <= t
            const int row = quad * 32 + lane, r = row >> 6, t = row & 63, hq = 2 * pr + r;
            float s[64];
            if (fac) {
                uint32_t r0[32], r1[32];
                tmem_ld32(tmem_addr(tmem + kOutSP, quad * 32, 0), r0);
                tmem_ld32(tmem_addr(tmem + kOutSP, quad * 32, 32), r1);
                tmem_ld_wait();
                reg_fence(r0);
                reg_fence(r1);
#pragma unroll
                for (int l = 0; l < 64; ++l) s[l] = l <= t ? __uint_as_float(l < 32 ? r0[l] : r1[l - 32]) : 0.f;
            } else {
                // one exponential per term: sum_k q_t[k] k_l[k] e^{G_t[k] - G_l[k]}
#pragma unroll
                for (int l = 0; l < 64; ++l) s[l] = 0.f;
                if (hq < G && ((vw >> t) & 1)) {
                    const __nv_bfloat16* qr = q + (((size_t)b * a.T + t0 + t) * a.Hq + (size_t)hk * G + hq) * kD;
#pragma unroll
                    for (int l = 0; l < 64; ++l) {
                        if (l > t || !((vw >> l) & 1)) continue;
                        const __nv_bfloat16* kr = kin + (((size_t)b * a.T + t0 + l) * a.Hkv + hk) * kD;
                        float acc = 0.f;
#pragma unroll 1
                        for (int k = 0; k < kD; ++k)
                            acc = fmaf(__bfloat162float(qr[k]) * __bfloat162float(kr[k]),
                                       __expf(Gs[t * kD + k] - Gs[l * kD + k]), acc);
                        s[l] = acc;
                    }
                }
            }
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                uint4 hi, lo;
                split8(s + 8 * cc, hi, lo);
                st16(Pp + swc(row, cc), hi);
                st16(Pp + 16384 + swc(row, cc), lo);
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            // Y = V^T P^T (rows v, columns (r, t))
#pragma unroll 1
            for (int ks = 0; ks < kC / 16; ++ks) {
                const uint64_t av = sdesc_sw128(smem_u32(Vt + ks * 2048), 8192, 1024);
                mma_ss(tmem + kOutY, av, sdesc_sw128(smem_u32(Pp + ks * 32), 16, 1024), idy, ks > 0);
                mma_ss(tmem + kOutY, av, sdesc_sw128(smem_u32(Pp + 16384 + ks * 32), 16, 1024), idy, 1);
            }
            mma_commit(bar_mma);
        }
        ok = warp_wait(bar_mma, mma_phase++ & 1, err, kErrMma);
        ok = __syncthreads_and(ok);
        if (!ok) break;
        tc_fence_after();
        {
            // outputs: warps 0-3 the pair's first head, warps 4-7 its second
            const int r = warp >> 2, v = quad * 32 + lane, hq = 2 * pr + r;
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                uint32_t rx[32], ry[32];
                tmem_ld32(tmem_addr(tmem + kOutX + 64 * r + 32 * half, quad * 32, 0), rx);
                tmem_ld32(tmem_addr(tmem + kOutY + 64 * r + 32 * half, quad * 32, 0), ry);
                tmem_ld_wait();
                reg_fence(rx);
                reg_fence(ry);
                if (hq < G) {
#pragma unroll
                    for (int x = 0; x < 32; ++x) {
                        const int t = 32 * half + x;
                        if (t0 + t >= a.T) continue;
                        const float o =
                            ((vw >> t) & 1) ? a.scale * (__uint_as_float(rx[x]) + __uint_as_float(ry[x])) : 0.f;
                        const size_t idx = (((size_t)b * a.T + t0 + t) * a.Hq + (size_t)hk * G + hq) * kD + v;
                        if (a.out_bf16)
                            reinterpret_cast<__nv_bfloat16*>(a.y)[idx] = __float2bfloat16_rn(o);
                        else
                            reinterpret_cast<float*>(a.y)[idx] = o;
                    }
                }
            }
        }
        tc_fence_before();
        __syncthreads();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace perdim

bool perdim_chunk_supported(const Problem& P) {
    if (!P.gated || P.delta || !P.decay_dim || !P.io_bf16 || P.Dk != perdim::kD || P.Dv != perdim::kD) return false;
    if (P.T < 1 || P.T > 0x7fffffffLL - 64) return false;
    const int64_t nc = (P.T + 63) / 64;
    return P.B * P.Hkv * nc <= 0x7fffffffLL && P.B * P.Hkv * perdim::kScanCtas <= 0x7fffffffLL;
}

size_t perdim_chunk_workspace_bytes(const Problem& P) {
    if (!perdim_chunk_supported(P)) return 0;
    return (size_t)P.B * P.Hkv * (size_t)((P.T + 63) / 64) * delta::Ws::kChunk;
}

cudaError_t perdim_chunk_causal(const Problem& P, const void* q, const void* k, const void* v, const void* decay,
                                const float* S0, void* y, float* S_out, void* ws, cudaStream_t st) {
    using namespace perdim;
    unsigned* err = device_error_word();
    if (!err) return cudaErrorInvalidDevice;
    static std::atomic<uint64_t> cfg_prep[kMaxDevices], cfg_out[kMaxDevices];
    cudaError_t e;
    if ((e = configure(perdim_prep_kernel, PrepSmem::kBytes, cfg_prep)) != cudaSuccess) return e;
    if ((e = configure(perdim_out_kernel, OutSmem::kBytes, cfg_out)) != cudaSuccess) return e;
    Args a;
    memset(&a, 0, sizeof(a));
    a.B = (int)P.B;
    a.T = (int)P.T;
    a.Hq = P.Hq;
    a.Hkv = P.Hkv;
    a.G = P.G;
    a.nc = (int)((P.T + 63) / 64);
    a.gated = 1;
    a.out_bf16 = P.out_bf16;
    a.scale = P.scale;
    a.decay = static_cast<const __nv_bfloat16*>(decay);
    a.mask = P.mask;
    a.S0 = S0;
    a.S_out = S_out;
    a.y = y;
    a.ws = static_cast<uint8_t*>(ws);
    a.err = err;
    if (!q || !k || !v || !a.decay || !a.y || !a.ws) return cudaErrorInvalidValue;  // every pointer the kernels use
    const unsigned streams = (unsigned)(P.B * P.Hkv);
    const unsigned chunks = streams * (unsigned)a.nc;
    perdim_prep_kernel<<<chunks, 128, PrepSmem::kBytes, st>>>(a, static_cast<const __nv_bfloat16*>(k),
                                                              static_cast<const __nv_bfloat16*>(v));
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    perdim_scan_kernel<<<streams * kScanCtas, kScanThreads, 0, st>>>(a);
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    perdim_out_kernel<<<chunks, 256, OutSmem::kBytes, st>>>(a, static_cast<const __nv_bfloat16*>(q),
                                                            static_cast<const __nv_bfloat16*>(k),
                                                            static_cast<const __nv_bfloat16*>(v));
    note_launch();
    return cudaGetLastError();
}

}  // namespace la
