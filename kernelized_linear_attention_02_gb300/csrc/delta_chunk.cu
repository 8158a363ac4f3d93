// delta_chunk.cu -- the delta rules of the ONNX-light "LinearAttention"
// operator (update rules "delta" and "gated_delta") in chunk-parallel form on
// the tensor cores (sm_103a: TMA, tcgen05, TMEM), for bf16 inputs with
// Dk = Dv = 128 and one log decay per kv head.
//
// The operator page allows chunk-parallel evaluation ("chunk_size: chunk size
// for the chunk-parallel WY decomposition during prefill").  Per (batch, kv
// head) stream and chunk of C = 64 steps with start state S0 (Dk x Dv), local
// steps t = 0..63, G_t the inclusive cumulative log decay inside the chunk,
// gamma_t = exp(G_t) and b_t = beta_t (a step that is masked out or past T has
// b = 0, g = 0 and zero key and value rows, so it changes nothing):
//
//   the rule S_t = e^{g_t} S_{t-1} + b_t k_t (v_t - e^{g_t} S_{t-1}^T k_t)^T
//   unrolls into S_t = gamma_t S0 + sum_{l<=t} (gamma_t / gamma_l) k_l u_l^T with
//     u_t = b_t (v_t - gamma_t S0^T k_t - sum_{l<t} (gamma_t/gamma_l)(k_t.k_l) u_l),
//   a unit lower-triangular system (I + A) U = diag(b) V - diag(b gamma) K S0,
//     A_tl = b_t (gamma_t / gamma_l) k_t.k_l  (l < t).
//   With T = (I + A)^{-1}, W = T diag(b gamma) K and U' = T diag(b) V:
//     U   = U' - W S0
//     S_C = gamma_C S0 + K^T diag(gamma_C / gamma) U = M S0 + N,
//           M = gamma_C I - K^T diag(gamma_C / gamma) W,  N = K^T diag(gamma_C / gamma) U'
//     O_r = diag(gamma) Q_r S0 + (Gamma o Q_r K^T) U,  Gamma_tl = gamma_t / gamma_l (l <= t)
//   (o_t = scale * S_t^T q_t for every query head r of the kv head).
//
// Three kernels, in stream order:
//   prep  one CTA per chunk, all chunks at once: T (blocked forward
//         substitution on CUDA cores), then W, U', M and N on the tensor cores
//   scan  S_{c+1} = M_c S_c + N_c, chunk after chunk, each stream's value
//         columns split over four CTAs; the start state of every chunk goes
//         to the workspace
//   out   one CTA per chunk: U and the outputs of every query head
// Every fp32 operand enters the tensor cores as bf16 hi + lo (about 16
// significant bits; products of the two lo parts are dropped); keys, values
// and queries are bf16 inputs and enter exactly.  All accumulation is fp32.
// Every wait is bounded: a wait that gives up records a bit in the device
// error word (la_device_error) and the kernel returns.
#include <algorithm>
#include <atomic>
#include <cstring>

#include "delta_args.h"
#include "kernels.h"
#include "tiles.cuh"
#include "tma_host.h"
#include "umma.cuh"

namespace la {
namespace delta {

using namespace umma;
using namespace tile;

constexpr int kC = 64;   // steps per chunk
constexpr int kD = 128;  // Dk = Dv
// Log decays below this are taken as this (exp of it underflows to zero in
// float32: a -inf step forgets everything before it, as the page's rule does).
constexpr float kMinLogDecay = -200.f;

// error bits of the delta kernels' bounded waits
enum : unsigned { kErrLoad = 1u << 16, kErrMma = 1u << 17 };



// Decay and update rate of steps 2 lane and 2 lane + 1 of chunk t0 (one warp):
// writes the inclusive cumulative log decay G_t and b_t (zero for steps that
// are masked out or past T) and returns the step-validity word.
__device__ __forceinline__ uint64_t chunk_steps(const Args& a, int b, int hk, int t0, float* Gs, float* Bs) {
    const int lane = threadIdx.x & 31;
    const int j0 = 2 * lane, j1 = j0 + 1;
    auto valid = [&](int j) {
        const int t = t0 + j;
        return t < a.T && (!a.mask || a.mask[(size_t)b * a.T + t] != 0);
    };
    const bool v0 = valid(j0), v1 = valid(j1);
    auto load_g = [&](int j) {
        return fmaxf(__bfloat162float(a.decay[((size_t)b * a.T + t0 + j) * a.Hkv + hk]), kMinLogDecay);
    };
    auto load_b = [&](int j) {
        const size_t bt = (size_t)b * a.T + t0 + j;
        return __bfloat162float(a.beta_per_head ? a.beta[bt * a.Hkv + hk] : a.beta[bt]);
    };
    const float g0 = (v0 && a.gated) ? load_g(j0) : 0.f, g1 = (v1 && a.gated) ? load_g(j1) : 0.f;
    const float sum = g0 + g1;
    float incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    Gs[j0] = incl - g1;
    Gs[j1] = incl;
    Bs[j0] = v0 ? load_b(j0) : 0.f;
    Bs[j1] = v1 ? load_b(j1) : 0.f;
    return step_word(v0, v1);
}

// ------------------------------------------------------------------ prep
// Shared memory of the prep kernel (offsets from the 1 KB-aligned base).
struct PrepSmem {
    static constexpr int kK = 0;          // K tile: 2 TMA boxes (k 0-63, 64-127) of 64 rows x 128 B
    static constexpr int kV = 16384;      // V tile
    static constexpr int kBw = 32768;     // T diag(b gamma) as B operand (rows t, K = l): hi, lo (8 KB each)
    static constexpr int kBu = 49152;     // T diag(b): hi, lo
    static constexpr int kBm = 65536;     // f_t W[t][k] as B operand (rows k, K = t): hi, lo (16 KB each)
    static constexpr int kAn = 98304;     // f_t U'[t][v] as A operand (rows v, K = t): hi, lo
    static constexpr int kA = 131072;     // A, fp32 [64][65]
    static constexpr int kT = kA + 64 * 65 * 4;   // T, fp32 [64][65]
    static constexpr int kX = kT + 64 * 65 * 4;   // [3][16][16] scratch of the blocked solve
    static constexpr int kGs = kX + 3 * 256 * 4;  // G_t [64]
    static constexpr int kBs = kGs + 256;         // b_t [64]
    static constexpr int kBar = kBs + 256;        // 2 mbarriers + TMEM slot
    static constexpr int kBytes = kBar + 64 + 1024;
};
// TMEM columns of the prep kernel
constexpr uint32_t kPrepKK = 0, kPrepW = 64, kPrepU = 128, kPrepM = 256, kPrepN = 384;

__global__ void __launch_bounds__(256, 1)
    delta_prep_kernel(const __grid_constant__ Args a, const __grid_constant__ CUtensorMap mK,
                      const __grid_constant__ CUtensorMap mV) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* Kt = sm + PrepSmem::kK;
    uint8_t* Vt = sm + PrepSmem::kV;
    uint8_t* Bw = sm + PrepSmem::kBw;
    uint8_t* Bu = sm + PrepSmem::kBu;
    uint8_t* Bm = sm + PrepSmem::kBm;
    uint8_t* An = sm + PrepSmem::kAn;
    float* Am = reinterpret_cast<float*>(sm + PrepSmem::kA);
    float* Tm = reinterpret_cast<float*>(sm + PrepSmem::kT);
    float* Xs = reinterpret_cast<float*>(sm + PrepSmem::kX);
    float* Gs = reinterpret_cast<float*>(sm + PrepSmem::kGs);
    float* Bs = reinterpret_cast<float*>(sm + PrepSmem::kBs);
    uint64_t* bar_ld = reinterpret_cast<uint64_t*>(sm + PrepSmem::kBar);
    uint64_t* bar_mma = bar_ld + 1;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bar_ld + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x / a.nc, c = blockIdx.x - bh * a.nc;
    const int b = bh / a.Hkv, hk = bh - b * a.Hkv;
    const int t0 = c * kC;
    uint8_t* wsc = a.ws + ((size_t)bh * a.nc + c) * Ws::kChunk;
    unsigned* err = a.err;

    if (tid == 0) {
        mbar_init(bar_ld, 1);
        mbar_init(bar_mma, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    bool ok = true;

    if (tid == 0) {
        tma_prefetch(&mK);
        tma_prefetch(&mV);
        mbar_arrive_expect_tx(bar_ld, 4 * 8192);
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_4d(Kt + kb * 8192, &mK, bar_ld, kb * 64, hk, t0, b);
            tma_load_4d(Vt + kb * 8192, &mV, bar_ld, kb * 64, hk, t0, b);
        }
    }
    uint64_t vword = 0;
    if (warp == 1) {
        vword = chunk_steps(a, b, hk, t0, Gs, Bs);
        float* wg = reinterpret_cast<float*>(wsc + Ws::kG);
        wg[2 * lane] = Gs[2 * lane];
        wg[2 * lane + 1] = Gs[2 * lane + 1];
        if (lane == 0) {
            wg[64] = __uint_as_float((uint32_t)vword);
            wg[65] = __uint_as_float((uint32_t)(vword >> 32));
        }
    }
    __shared__ uint64_t s_vword;
    if (tid == 32) s_vword = vword;
    ok = warp_wait(bar_ld, 0, err, kErrLoad);
    ok = __syncthreads_and(ok);
    vword = s_vword;
    // masked-out steps inside T: zero key and value rows (rows past T arrive
    // as zeros from the tensor map)
    if (a.mask) {
        const int nvalid = min(kC, a.T - t0);
        const uint64_t inside = nvalid >= 64 ? ~0ull : ((1ull << nvalid) - 1);
        if ((vword & inside) != inside) {
            for (int e = tid; e < 64 * 32; e += 256) {
                const int r = e >> 5, q = e & 31;  // q: tile (K/V), K block, 16-byte chunk
                if (r < nvalid && !((vword >> r) & 1)) {
                    uint8_t* tile = (q < 16 ? Kt : Vt) + ((q >> 3) & 1) * 8192;
                    st16(tile + swc(r, q & 7), make_uint4(0, 0, 0, 0));
                }
            }
            fence_proxy_async();
        }
    }
    __syncthreads();

    // ---- K K^T (M = 64: rows t in TMEM lanes 0-15 of each quadrant)
    if (tid == 0 && ok) {
        tc_fence_after();
        constexpr uint32_t id = idesc_bf16(64, 64, false, false);
#pragma unroll 1
        for (int ks = 0; ks < kD / 16; ++ks) {
            const uint64_t d = sdesc_sw128(smem_u32(Kt + (ks >> 2) * 8192 + (ks & 3) * 32), 16, 1024);
            mma_ss(tmem + kPrepKK, d, d, id, ks > 0);
        }
        mma_commit(bar_mma);
    }
    if (ok) ok = warp_wait(bar_mma, 0, err, kErrMma);
    tc_fence_after();
    if (warp < 4) {
        // A_tl = b_t exp(G_t - G_l) k_t.k_l for l < t; this thread holds rows
        // r1 = 16 quad + lane/4 and r2 = r1 + 8, columns 8g + cq and + 1
        const int quad = warp;
        uint32_t sc[32];
        tmem_ld16x256b_x8(tmem_addr(tmem + kPrepKK, quad * 32, 0), sc);
        tmem_ld_wait();
        reg_fence(sc);
        const int r1 = quad * 16 + (lane >> 2), r2 = r1 + 8, cq = 2 * (lane & 3);
        const float g1 = Gs[r1], g2 = Gs[r2], b1 = Bs[r1], b2 = Bs[r2];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int j = 8 * g + cq + e;
                Am[r1 * 65 + j] = j < r1 ? b1 * __expf(g1 - Gs[j]) * __uint_as_float(sc[4 * g + e]) : 0.f;
                Am[r2 * 65 + j] = j < r2 ? b2 * __expf(g2 - Gs[j]) * __uint_as_float(sc[4 * g + 2 + e]) : 0.f;
            }
        }
    } else {
        for (int e = tid - 128; e < 64 * 65; e += 128) Tm[e] = 0.f;
    }
    __syncthreads();

    // ---- T = (I + A)^{-1}: 16 x 16 diagonal blocks by forward substitution
    // (one warp per block, lane j < 16 one column), then the blocks below the
    // diagonal level by level: T_ij = -T_ii sum_{j <= k < i} A_ik T_kj
    if (warp < 4 && lane < 16) {
        const int o = 16 * warp, j = lane;
        float tc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float acc = 0.f;
#pragma unroll
            for (int l = 0; l < i; ++l) acc = fmaf(Am[(o + i) * 65 + o + l], tc[l], acc);
            tc[i] = i < j ? 0.f : (i == j ? 1.f : -acc);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) Tm[(o + i) * 65 + o + j] = tc[i];
    }
    __syncthreads();
#pragma unroll 1
    for (int d = 1; d < 4; ++d) {
        const int nblk = 4 - d;  // blocks (i, i - d), i = d..3
        for (int e = tid; e < nblk * 256; e += 256) {
            const int bi = d + e / 256, bj = bi - d, r = (e >> 4) & 15, cl = e & 15;
            float acc = 0.f;
            for (int col = 16 * bj; col < 16 * bi; ++col) acc = fmaf(Am[(16 * bi + r) * 65 + col], Tm[col * 65 + 16 * bj + cl], acc);
            Xs[e] = acc;
        }
        __syncthreads();
        for (int e = tid; e < nblk * 256; e += 256) {
            const int bi = d + e / 256, bj = bi - d, r = (e >> 4) & 15, cl = e & 15;
            const float* x = Xs + (e / 256) * 256;
            float acc = 0.f;
#pragma unroll
            for (int cc = 0; cc < 16; ++cc) acc = fmaf(Tm[(16 * bi + r) * 65 + 16 * bi + cc], x[cc * 16 + cl], acc);
            Tm[(16 * bi + r) * 65 + 16 * bj + cl] = -acc;
        }
        __syncthreads();
    }

    // ---- B operands T diag(b gamma) and T diag(b) (rows t, K = l), hi + lo
    for (int e = tid; e < 64 * 8; e += 256) {
        const int t = e >> 3, cc = e & 7;
        float fw[8], fu[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            const int l = 8 * cc + x;
            const float tv = Tm[t * 65 + l] * Bs[l];
            fu[x] = tv;
            fw[x] = tv * __expf(Gs[l]);
        }
        uint4 hi, lo;
        split8(fw, hi, lo);
        st16(Bw + swc(t, cc), hi);
        st16(Bw + 8192 + swc(t, cc), lo);
        split8(fu, hi, lo);
        st16(Bu + swc(t, cc), hi);
        st16(Bu + 8192 + swc(t, cc), lo);
    }
    fence_proxy_async();
    __syncthreads();

    // ---- W^T (rows k) = K^T (T diag(b gamma))^T and U'^T (rows v) = V^T (T diag(b))^T
    if (tid == 0 && ok) {
        tc_fence_after();
        constexpr uint32_t id = idesc_bf16(128, 64, true, false);
#pragma unroll 1
        for (int ks = 0; ks < kC / 16; ++ks) {
            const uint64_t ak = sdesc_sw128(smem_u32(Kt + ks * 2048), 8192, 1024);
            const uint64_t av = sdesc_sw128(smem_u32(Vt + ks * 2048), 8192, 1024);
            mma_ss(tmem + kPrepW, ak, sdesc_sw128(smem_u32(Bw + ks * 32), 16, 1024), id, ks > 0);
            mma_ss(tmem + kPrepW, ak, sdesc_sw128(smem_u32(Bw + 8192 + ks * 32), 16, 1024), id, 1);
            mma_ss(tmem + kPrepU, av, sdesc_sw128(smem_u32(Bu + ks * 32), 16, 1024), id, ks > 0);
            mma_ss(tmem + kPrepU, av, sdesc_sw128(smem_u32(Bu + 8192 + ks * 32), 16, 1024), id, 1);
        }
        mma_commit(bar_mma);
    }
    if (ok) ok = warp_wait(bar_mma, 1, err, kErrMma);
    tc_fence_after();
    {
        const int quad = warp & 3, row = quad * 32 + lane;  // k (warps 0-3) or v (warps 4-7)
        const bool wside = warp < 4;
        uint32_t r0[32], r1[32];
        const uint32_t col = wside ? kPrepW : kPrepU;
        tmem_ld32(tmem_addr(tmem + col, quad * 32, 0), r0);
        tmem_ld32(tmem_addr(tmem + col, quad * 32, 32), r1);
        tmem_ld_wait();
        reg_fence(r0);
        reg_fence(r1);
        const float gC = Gs[kC - 1];
        auto val = [&](int t) { return __uint_as_float(t < 32 ? r0[t] : r1[t - 32]); };
        if (wside) {
            // W[t][k] to the workspace (B operand of the output kernel: rows t,
            // K = k), and f_t W[t][k] as this row k of the B operand of M
            __nv_bfloat16* wh = reinterpret_cast<__nv_bfloat16*>(wsc + Ws::kW);
            const int kb = row >> 6, kc = row & 63;
#pragma unroll
            for (int t = 0; t < 64; ++t) {
                const float x = val(t);
                const __nv_bfloat16 h = __float2bfloat16_rn(x);
                const uint32_t off = kb * 8192 + swe(t, kc);
                *reinterpret_cast<__nv_bfloat16*>(reinterpret_cast<uint8_t*>(wh) + off) = h;
                *reinterpret_cast<__nv_bfloat16*>(reinterpret_cast<uint8_t*>(wh) + 16384 + off) =
                    __float2bfloat16_rn(x - __bfloat162float(h));
            }
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                float f[8];
#pragma unroll
                for (int x = 0; x < 8; ++x) f[x] = __expf(gC - Gs[8 * cc + x]) * val(8 * cc + x);
                uint4 hi, lo;
                split8(f, hi, lo);
                st16(Bm + swc(row, cc), hi);
                st16(Bm + 16384 + swc(row, cc), lo);
            }
        } else {
            // U'[t][v] to the workspace, and f_t U'[t][v] as row v of the A operand of N^T
            float* up = reinterpret_cast<float*>(wsc + Ws::kU);
#pragma unroll
            for (int t = 0; t < 64; ++t) up[t * kD + row] = val(t);
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                float f[8];
#pragma unroll
                for (int x = 0; x < 8; ++x) f[x] = __expf(gC - Gs[8 * cc + x]) * val(8 * cc + x);
                uint4 hi, lo;
                split8(f, hi, lo);
                st16(An + swc(row, cc), hi);
                st16(An + 16384 + swc(row, cc), lo);
            }
        }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // ---- M (rows k') = K^T (f W) ... as D[k'][k] = sum_t K[t][k'] f_t W[t][k],
    // and N^T (rows v) = (f U')^T K
    if (tid == 0 && ok) {
        tc_fence_after();
        constexpr uint32_t idm = idesc_bf16(128, 128, true, false);
        constexpr uint32_t idn = idesc_bf16(128, 128, false, true);
#pragma unroll 1
        for (int ks = 0; ks < kC / 16; ++ks) {
            const uint64_t ak = sdesc_sw128(smem_u32(Kt + ks * 2048), 8192, 1024);  // also N^T's B
            mma_ss(tmem + kPrepM, ak, sdesc_sw128(smem_u32(Bm + ks * 32), 16, 1024), idm, ks > 0);
            mma_ss(tmem + kPrepM, ak, sdesc_sw128(smem_u32(Bm + 16384 + ks * 32), 16, 1024), idm, 1);
            mma_ss(tmem + kPrepN, sdesc_sw128(smem_u32(An + ks * 32), 16, 1024), ak, idn, ks > 0);
            mma_ss(tmem + kPrepN, sdesc_sw128(smem_u32(An + 16384 + ks * 32), 16, 1024), ak, idn, 1);
        }
        mma_commit(bar_mma);
    }
    if (ok) ok = warp_wait(bar_mma, 0, err, kErrMma);
    tc_fence_after();
    {
        const int quad = warp & 3, row = quad * 32 + lane;
        const float gammaC = __expf(Gs[kC - 1]);
        if (warp < 4) {
            // row k' of M = gamma_C I - D, to the workspace (A operand of the
            // scan: rows k', K = k), hi + lo
            uint8_t* mt = wsc + Ws::kM;
#pragma unroll 1
            for (int p = 0; p < 4; ++p) {
                uint32_t r[32];
                tmem_ld32(tmem_addr(tmem + kPrepM, quad * 32, 32 * p), r);
                tmem_ld_wait();
                reg_fence(r);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    float f[8];
#pragma unroll
                    for (int x = 0; x < 8; ++x) {
                        const int k = 32 * p + 8 * q4 + x;
                        f[x] = (k == row ? gammaC : 0.f) - __uint_as_float(r[8 * q4 + x]);
                    }
                    uint4 hi, lo;
                    split8(f, hi, lo);
                    const int k0 = 32 * p + 8 * q4;
                    const uint32_t off = (k0 >> 6) * 16384 + swc(row, (k0 & 63) >> 3);
                    st16(mt + off, hi);
                    st16(mt + 32768 + off, lo);
                }
            }
        } else {
            // row v of N^T, stored as N [k][v] fp32
            float* nt = reinterpret_cast<float*>(wsc + Ws::kN);
#pragma unroll 1
            for (int p = 0; p < 4; ++p) {
                uint32_t r[32];
                tmem_ld32(tmem_addr(tmem + kPrepN, quad * 32, 32 * p), r);
                tmem_ld_wait();
                reg_fence(r);
#pragma unroll
                for (int x = 0; x < 32; ++x) nt[(32 * p + x) * kD + row] = __uint_as_float(r[x]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ scan
// The columns of the state are independent under S <- M S + N (M acts on the
// key dimension), so each stream's scan is split over kScanSplit CTAs of
// kScanV value columns each: per chunk the CTA computes its block of M_c S_c
// (M = 128 keys, N = kScanV values, K = 128) on the tensor cores, adds N_c in
// fp32 and writes the next start state as the B operand of the next chunk's
// product.  The smaller product and epilogue shorten the chunk-to-chunk chain.
constexpr int kScanV = 32;                 // value columns per CTA
constexpr int kScanSplit = kD / kScanV;    // CTAs per stream
struct ScanSmem {
    static constexpr int kM = 0;           // two M stages of 64 KB (A operand, rows k'; hi 32 KB, lo 32 KB)
    static constexpr int kB = 131072;      // S block as B operand (rows v, K = k): hi 8 KB, lo 8 KB
    static constexpr int kBar = kB + 16384;  // mfull[2], mma, TMEM slot
    static constexpr int kBytes = kBar + 64 + 1024;
};

__global__ void __launch_bounds__(128, 1) delta_scan_kernel(const __grid_constant__ Args a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* Mr = sm + ScanSmem::kM;
    uint8_t* Bt = sm + ScanSmem::kB;
    uint64_t* mfull = reinterpret_cast<uint64_t*>(sm + ScanSmem::kBar);  // [2]
    uint64_t* bar_mma = mfull + 2;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mfull + 3);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int bh = blockIdx.x / kScanSplit, v0 = kScanV * (blockIdx.x - bh * kScanSplit);
    const int nc = a.nc;
    const int kr = tid;  // key row k' of the product held by this thread (TMEM lane)
    uint8_t* ws0 = a.ws + (size_t)bh * nc * Ws::kChunk;
    unsigned* err = a.err;

    if (tid == 0) {
        mbar_init(&mfull[0], 1);
        mbar_init(&mfull[1], 1);
        mbar_init(bar_mma, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, 32);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    if (tid == 0) {
        for (int c = 0; c < min(2, nc); ++c) {
            mbar_arrive_expect_tx(&mfull[c], 65536);
            bulk_load(Mr + c * 65536, ws0 + (size_t)c * Ws::kChunk + Ws::kM, 65536, &mfull[c]);
        }
    }
    // S[k'][v0 .. v0 + 31] as column k' of the B tile (row v, K = k'), hi and lo
    auto put_block = [&](const float (&s)[kScanV]) {
        const uint32_t base = (kr >> 6) * 4096;
#pragma unroll
        for (int x = 0; x < kScanV; ++x) {
            const __nv_bfloat16 h = __float2bfloat16_rn(s[x]);
            const uint32_t off = base + swe(x, kr & 63);
            *reinterpret_cast<__nv_bfloat16*>(Bt + off) = h;
            *reinterpret_cast<__nv_bfloat16*>(Bt + 8192 + off) = __float2bfloat16_rn(s[x] - __bfloat162float(h));
        }
    };
    auto load_row = [&](const float* src, float (&s)[kScanV]) {  // 32 consecutive floats, 16-byte aligned
#pragma unroll
        for (int x = 0; x < kScanV; x += 4) {
            const float4 f = *reinterpret_cast<const float4*>(src + x);
            s[x] = f.x, s[x + 1] = f.y, s[x + 2] = f.z, s[x + 3] = f.w;
        }
    };
    {
        float s[kScanV];  // (the state pointers are only 4-byte aligned)
        const float* s0 = a.S0 ? a.S0 + (size_t)bh * kD * kD + (size_t)kr * kD + v0 : nullptr;
#pragma unroll
        for (int x = 0; x < kScanV; ++x) s[x] = s0 ? s0[x] : 0.f;
        put_block(s);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    bool ok = true;
    constexpr uint32_t id = idesc_bf16(128, kScanV, false, false);
#pragma unroll 1
    for (int c = 0; c < nc; ++c) {
        uint8_t* wsc = ws0 + (size_t)c * Ws::kChunk;
        bool mok = true;  // M_c arrived (thread 0)
        if (tid == 0) {
            tc_fence_after();
            // the start state of chunk c (rows v0 .. v0 + 31 of each K block of its S^T tile)
#pragma unroll
            for (int part = 0; part < 4; ++part) {  // (hi, lo) x K block
                const int kb = part & 1, lo = part >> 1;
                bulk_store(wsc + Ws::kS + lo * 32768 + kb * 16384 + v0 * 128, Bt + lo * 8192 + kb * 4096, 4096);
            }
            bulk_commit_group();
            // M_c S_c: A = M_c (rows k', K = k), B = S_c block (rows v, K = k)
            mok = mbar_wait(&mfull[c & 1], (c >> 1) & 1, err, kErrLoad);
            if (mok) {
                const uint8_t* mt = Mr + (c & 1) * 65536;
#pragma unroll 1
                for (int ks = 0; ks < kD / 16; ++ks) {
                    const uint32_t ao = (ks >> 2) * 16384 + (ks & 3) * 32;
                    const uint32_t bo = (ks >> 2) * 4096 + (ks & 3) * 32;
                    const uint64_t ah = sdesc_sw128(smem_u32(mt + ao), 16, 1024);
                    const uint64_t al = sdesc_sw128(smem_u32(mt + 32768 + ao), 16, 1024);
                    const uint64_t bh_ = sdesc_sw128(smem_u32(Bt + bo), 16, 1024);
                    const uint64_t bl_ = sdesc_sw128(smem_u32(Bt + 8192 + bo), 16, 1024);
                    mma_ss(tmem, ah, bh_, id, ks > 0);
                    mma_ss(tmem, ah, bl_, id, 1);
                    mma_ss(tmem, al, bh_, id, 1);
                }
            }
            mma_commit(bar_mma);
        }
        // N_c[k'][v0 .. v0 + 31] while the product runs
        float n[kScanV];
        load_row(reinterpret_cast<const float*>(wsc + Ws::kN) + (size_t)kr * kD + v0, n);
        ok = warp_wait(bar_mma, c & 1, err, kErrMma) && mok;
        if (tid == 0) {
            if (ok && c + 2 < nc) {  // stage c & 1 is free: M of chunk c + 2
                mbar_arrive_expect_tx(&mfull[c & 1], 65536);
                bulk_load(Mr + (c & 1) * 65536, ws0 + (size_t)(c + 2) * Ws::kChunk + Ws::kM, 65536, &mfull[c & 1]);
            }
            bulk_wait_group_read<0>();  // the B tile has been copied out
        }
        ok = __syncthreads_and(ok);  // every exit below is taken by the whole block
        if (!ok) break;
        tc_fence_after();
        uint32_t r[32];
        tmem_ld32(tmem_addr(tmem, warp * 32, 0), r);
        tmem_ld_wait();
        reg_fence(r);
        float s[kScanV];
#pragma unroll
        for (int x = 0; x < kScanV; ++x) s[x] = __uint_as_float(r[x]) + n[x];
        if (c + 1 < nc) {
            put_block(s);
        } else if (a.S_out) {
            float* dst = a.S_out + (size_t)bh * kD * kD + (size_t)kr * kD + v0;
#pragma unroll
            for (int x = 0; x < kScanV; ++x) dst[x] = s[x];
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
    }
    if (tid == 0) bulk_wait_group<0>();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 32);
    }
}

// ------------------------------------------------------------------ out
struct OutSmem {
    static constexpr int kS = 0;          // S_c^T as A operand (rows v, K = k): hi 32 KB, lo 32 KB
    static constexpr int kW = 65536;      // W as B operand (rows t, K = k): hi 16 KB, lo 16 KB
    static constexpr int kK = 98304;      // K tile (rows l, K = k), 2 TMA boxes
    static constexpr int kQ = 114688;     // two query heads (rows (r, t), K = k): block kb at kb * 16 KB, head r at + 8 KB
    static constexpr int kUa = 147456;    // U^T as A operand (rows v, K = t): hi, lo (16 KB each)
    static constexpr int kP = 180224;     // P as B operand (rows (r, t), K = l): hi, lo (16 KB each)
    static constexpr int kGs = 212992;    // G_t [64]
    static constexpr int kBar = kGs + 256;
    static constexpr int kBytes = kBar + 64 + 1024;
};
constexpr uint32_t kOutU = 0, kOutSP = 64, kOutX = 128, kOutY = 256;

__global__ void __launch_bounds__(256, 1)
    delta_out_kernel(const __grid_constant__ Args a, const __grid_constant__ CUtensorMap mQ,
                     const __grid_constant__ CUtensorMap mK) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* St = sm + OutSmem::kS;
    uint8_t* Wt = sm + OutSmem::kW;
    uint8_t* Kt = sm + OutSmem::kK;
    uint8_t* Qp = sm + OutSmem::kQ;
    uint8_t* Ua = sm + OutSmem::kUa;
    uint8_t* Pp = sm + OutSmem::kP;
    float* Gs = reinterpret_cast<float*>(sm + OutSmem::kGs);
    uint64_t* bar_ld = reinterpret_cast<uint64_t*>(sm + OutSmem::kBar);
    uint64_t* bar_mma = bar_ld + 1;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bar_ld + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x / a.nc, c = blockIdx.x - bh * a.nc;
    const int b = bh / a.Hkv, hk = bh - b * a.Hkv;
    const int t0 = c * kC, G = a.G;
    const uint8_t* wsc = a.ws + ((size_t)bh * a.nc + c) * Ws::kChunk;
    unsigned* err = a.err;

    if (tid == 0) {
        mbar_init(bar_ld, 1);
        mbar_init(bar_mma, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    uint32_t ld_phase = 0, mma_phase = 0;
    auto load_pair = [&](int pr, uint32_t extra) {  // query heads 2 pr and 2 pr + 1 of this kv head
        mbar_arrive_expect_tx(bar_ld, 4 * 8192 + extra);
        for (int r = 0; r < 2; ++r)
            for (int kb = 0; kb < 2; ++kb)
                tma_load_4d(Qp + kb * 16384 + r * 8192, &mQ, bar_ld, kb * 64, hk * G + 2 * pr + r, t0, b);
    };
    if (tid == 0) {
        tma_prefetch(&mQ);
        tma_prefetch(&mK);
        load_pair(0, 65536 + 32768 + 2 * 8192);
        bulk_load(St, wsc + Ws::kS, 65536, bar_ld);
        bulk_load(Wt, wsc + Ws::kW, 32768, bar_ld);
        for (int kb = 0; kb < 2; ++kb) tma_load_4d(Kt + kb * 8192, &mK, bar_ld, kb * 64, hk, t0, b);
    }
    const float* wg = reinterpret_cast<const float*>(wsc + Ws::kG);
    if (tid < 64) Gs[tid] = wg[tid];
    const uint64_t vword = (uint64_t)__float_as_uint(wg[64]) | ((uint64_t)__float_as_uint(wg[65]) << 32);
    // U'^T row v (warps 0-3), in flight while the loads and the first products run
    float upre[kC];
    if (warp < 4) {
        const float* up = reinterpret_cast<const float*>(wsc + Ws::kU);
        const int v = (warp & 3) * 32 + lane;
#pragma unroll
        for (int t = 0; t < kC; ++t) upre[t] = up[t * kD + v];
    }
    bool ok = warp_wait(bar_ld, ld_phase++ & 1, err, kErrLoad);
    ok = __syncthreads_and(ok);

    constexpr uint32_t id64 = idesc_bf16(128, 64, false, false);
    constexpr uint32_t id128 = idesc_bf16(128, 128, false, false);
    // scores of the current head pair: rows (r, t), columns l
    auto issue_scores = [&]() {
#pragma unroll 1
        for (int ks = 0; ks < kD / 16; ++ks) {
            const uint64_t aq = sdesc_sw128(smem_u32(Qp + (ks >> 2) * 16384 + (ks & 3) * 32), 16, 1024);
            const uint64_t bk = sdesc_sw128(smem_u32(Kt + (ks >> 2) * 8192 + (ks & 3) * 32), 16, 1024);
            mma_ss(tmem + kOutSP, aq, bk, id64, ks > 0);
        }
    };
    if (tid == 0 && ok) {
        tc_fence_after();
        // U^T - U'^T = -(S^T W^T): A = S^T (rows v), B = W (rows t)
#pragma unroll 1
        for (int ks = 0; ks < kD / 16; ++ks) {
            const uint32_t ao = (ks >> 2) * 16384 + (ks & 3) * 32, bo = (ks >> 2) * 8192 + (ks & 3) * 32;
            const uint64_t ah = sdesc_sw128(smem_u32(St + ao), 16, 1024), al = sdesc_sw128(smem_u32(St + 32768 + ao), 16, 1024);
            const uint64_t bh_ = sdesc_sw128(smem_u32(Wt + bo), 16, 1024), bl_ = sdesc_sw128(smem_u32(Wt + 16384 + bo), 16, 1024);
            mma_ss(tmem + kOutU, ah, bh_, id64, ks > 0);
            mma_ss(tmem + kOutU, ah, bl_, id64, 1);
            mma_ss(tmem + kOutU, al, bh_, id64, 1);
        }
        issue_scores();
        mma_commit(bar_mma);
    }
    if (ok) ok = warp_wait(bar_mma, mma_phase++ & 1, err, kErrMma);
    ok = __syncthreads_and(ok);
    tc_fence_after();
    const int quad = warp & 3;
    // P rows (r, t): exp(G_t - G_l) q_t.k_l for l <= t (warps 4-7)
    auto make_p = [&]() {
        const int row = quad * 32 + lane, t = row & 63;
        uint32_t r0[32], r1[32];
        tmem_ld32(tmem_addr(tmem + kOutSP, quad * 32, 0), r0);
        tmem_ld32(tmem_addr(tmem + kOutSP, quad * 32, 32), r1);
        tmem_ld_wait();
        reg_fence(r0);
        reg_fence(r1);
        const float gt = Gs[t];
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
            float f[8];
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                const int l = 8 * cc + x;
                const float sv = __uint_as_float(l < 32 ? r0[l] : r1[l - 32]);
                f[x] = l <= t ? sv * __expf(gt - Gs[l]) : 0.f;
            }
            uint4 hi, lo;
            split8(f, hi, lo);
            st16(Pp + swc(row, cc), hi);
            st16(Pp + 16384 + swc(row, cc), lo);
        }
    };
    if (warp < 4) {
        // U^T row v = U'^T - acc, hi/lo as row v of the A operand of Y
        const int v = quad * 32 + lane;
        uint32_t r0[32], r1[32];
        tmem_ld32(tmem_addr(tmem + kOutU, quad * 32, 0), r0);
        tmem_ld32(tmem_addr(tmem + kOutU, quad * 32, 32), r1);
        tmem_ld_wait();
        reg_fence(r0);
        reg_fence(r1);
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
            float f[8];
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                const int t = 8 * cc + x;
                f[x] = upre[t] - __uint_as_float(t < 32 ? r0[t] : r1[t - 32]);
            }
            uint4 hi, lo;
            split8(f, hi, lo);
            st16(Ua + swc(v, cc), hi);
            st16(Ua + 16384 + swc(v, cc), lo);
        }
    } else {
        make_p();
    }
    const int npairs = (G + 1) / 2;
    // (ok is uniform across the block here and after every __syncthreads_and)
#pragma unroll 1
    for (int pr = 0; pr < npairs && ok; ++pr) {
        if (pr > 0) {
            // next head pair: its queries were requested when the previous
            // pair's products completed; then scores and P
            tc_fence_before();
            __syncthreads();
            ok = warp_wait(bar_ld, ld_phase++ & 1, err, kErrLoad);
            ok = __syncthreads_and(ok);
            if (!ok) break;
            if (tid == 0) {
                tc_fence_after();
                issue_scores();
                mma_commit(bar_mma);
            }
            ok = warp_wait(bar_mma, mma_phase++ & 1, err, kErrMma);
            ok = __syncthreads_and(ok);
            if (!ok) break;
            tc_fence_after();
            if (warp >= 4) make_p();
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            // X = S^T Q^T (rows v, columns (r, t)) and Y = U^T P^T
#pragma unroll 1
            for (int ks = 0; ks < kD / 16; ++ks) {
                const uint32_t ao = (ks >> 2) * 16384 + (ks & 3) * 32;
                const uint64_t bq = sdesc_sw128(smem_u32(Qp + ao), 16, 1024);
                mma_ss(tmem + kOutX, sdesc_sw128(smem_u32(St + ao), 16, 1024), bq, id128, ks > 0);
                mma_ss(tmem + kOutX, sdesc_sw128(smem_u32(St + 32768 + ao), 16, 1024), bq, id128, 1);
            }
#pragma unroll 1
            for (int ks = 0; ks < kC / 16; ++ks) {
                const uint64_t ah = sdesc_sw128(smem_u32(Ua + ks * 32), 16, 1024);
                const uint64_t al = sdesc_sw128(smem_u32(Ua + 16384 + ks * 32), 16, 1024);
                const uint64_t bh_ = sdesc_sw128(smem_u32(Pp + ks * 32), 16, 1024);
                const uint64_t bl_ = sdesc_sw128(smem_u32(Pp + 16384 + ks * 32), 16, 1024);
                mma_ss(tmem + kOutY, ah, bh_, id128, ks > 0);
                mma_ss(tmem + kOutY, ah, bl_, id128, 1);
                mma_ss(tmem + kOutY, al, bh_, id128, 1);
            }
            mma_commit(bar_mma);
        }
        ok = warp_wait(bar_mma, mma_phase++ & 1, err, kErrMma);
        ok = __syncthreads_and(ok);
        if (!ok) break;
        tc_fence_after();
        // the products have read this pair's queries: the next pair's load overlaps the outputs
        if (tid == 0 && pr + 1 < npairs) load_pair(pr + 1, 0);
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
                        const float o = ((vword >> t) & 1)
                                            ? a.scale * (__expf(Gs[t]) * __uint_as_float(rx[x]) + __uint_as_float(ry[x]))
                                            : 0.f;
                        const size_t idx = (((size_t)b * a.T + t0 + t) * a.Hq + (size_t)hk * G + hq) * kD + v;
                        if (a.out_bf16)
                            reinterpret_cast<__nv_bfloat16*>(a.y)[idx] = __float2bfloat16_rn(o);
                        else
                            reinterpret_cast<float*>(a.y)[idx] = o;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace delta

bool delta_chunk_supported(const Problem& P) {
    if (!P.delta || !P.io_bf16 || P.Dk != delta::kD || P.Dv != delta::kD || P.decay_dim) return false;
    if (P.T < 1 || P.T > 0x7fffffffLL - 64) return false;
    const int64_t nc = (P.T + 63) / 64;
    return P.B * P.Hkv * nc <= 0x7fffffffLL && P.B * P.Hkv * delta::kScanSplit <= 0x7fffffffLL;
}

size_t delta_chunk_workspace_bytes(const Problem& P) {
    if (!delta_chunk_supported(P)) return 0;
    return (size_t)P.B * P.Hkv * (size_t)((P.T + 63) / 64) * delta::Ws::kChunk;
}

cudaError_t delta_chunk_causal(const Problem& P, const void* q, const void* k, const void* v, const void* decay,
                               const void* beta, int beta_per_head, const float* S0, void* y, float* S_out,
                               void* ws, cudaStream_t st) {
    using namespace delta;
    unsigned* err = device_error_word();
    if (!err) return cudaErrorInvalidDevice;
    static std::atomic<uint64_t> cfg_prep[kMaxDevices], cfg_scan[kMaxDevices], cfg_out[kMaxDevices];
    cudaError_t e;
    if ((e = configure(delta_prep_kernel, PrepSmem::kBytes, cfg_prep)) != cudaSuccess) return e;
    if ((e = configure(delta_scan_kernel, ScanSmem::kBytes, cfg_scan)) != cudaSuccess) return e;
    if ((e = configure(delta_out_kernel, OutSmem::kBytes, cfg_out)) != cudaSuccess) return e;
    CUtensorMap mq, mk, mv;
    if (!act_map(&mq, q, P.Hq, P.T, P.B) || !act_map(&mk, k, P.Hkv, P.T, P.B) || !act_map(&mv, v, P.Hkv, P.T, P.B))
        return cudaErrorInvalidValue;
    Args a;
    memset(&a, 0, sizeof(a));
    a.B = (int)P.B;
    a.T = (int)P.T;
    a.Hq = P.Hq;
    a.Hkv = P.Hkv;
    a.G = P.G;
    a.nc = (int)((P.T + 63) / 64);
    a.gated = P.gated;
    a.beta_per_head = beta_per_head;
    a.out_bf16 = P.out_bf16;
    a.scale = P.scale;
    a.decay = static_cast<const __nv_bfloat16*>(decay);
    a.beta = static_cast<const __nv_bfloat16*>(beta);
    a.mask = P.mask;
    a.S0 = S0;
    a.S_out = S_out;
    a.y = y;
    a.ws = static_cast<uint8_t*>(ws);
    a.err = err;
    if (!a.beta || !a.y || !a.ws || (a.gated && !a.decay)) return cudaErrorInvalidValue;  // every pointer the kernels use
    const unsigned streams = (unsigned)(P.B * P.Hkv);
    const unsigned chunks = streams * (unsigned)a.nc;
    delta_prep_kernel<<<chunks, 256, PrepSmem::kBytes, st>>>(a, mk, mv);
    delta_scan_kernel<<<streams * kScanSplit, 128, ScanSmem::kBytes, st>>>(a);
    delta_out_kernel<<<chunks, 256, OutSmem::kBytes, st>>>(a, mq, mk);
    note_launch(3);
    return cudaGetLastError();
}


}  // namespace la
