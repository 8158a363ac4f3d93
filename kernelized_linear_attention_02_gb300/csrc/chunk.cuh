// chunk.cuh -- the chunk-parallel tensor-core kernel for bf16 inputs
// (sm_103a: TMA + tcgen05 + TMEM), instantiated per head size in
// chunk_d64.cu / chunk_d128.cu.
//
// Causal form per chunk of C = 64 tokens (Keras request, "Mathematical
// definition / Causal"; ONNX LinearAttention "may be implemented using
// chunk-parallel algorithms"), written transposed so that the value
// dimension is the MMA's M (= Dv) and the state never leaves tensor memory:
//
//   Y^T   = S_prev^T . phi(Q)^T                    (inter-chunk read-out)
//         + V^T . mask(phi(Q) phi(K)^T)^T          (intra-chunk, j <= i)
//   den_i = phi(q_i).Z_prev + sum_{j<=i} phi(q_i).phi(k_j) + eps
//   S^T  += V^T . phi(K)                           (state carry, fp32)
//   Z    += sum_j phi(k_j)
//
// Gated rule (ONNX "gated", per-head scalar log decay g): with G_i the
// inclusive cumulative sum of g inside the chunk, the read-out uses
// exp(G_i) q_i against S_prev, the intra weights are multiplied by
// exp(G_i - G_j) (<= 1), and the carry is S <- exp(G_C) S + sum_j
// exp(G_C - G_j) k_j v_j^T.
//
// Precision: phi(Q) and phi(K) enter the tensor cores as bf16; the masked
// score matrix and the carried state are split into bf16 hi + lo parts, so
// that both reach the tensor cores with ~16 significant bits; the state
// update uses a hi + lo split of the key operand whenever phi(k) (or the
// decayed key) is not exactly representable in bf16.  All accumulation is
// fp32 in tensor memory.
//
// Roles (320 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM
// owner, warps 2-5 operand converters (feature map, hi/lo splits, Z, state
// hi/lo in TMEM), warps 6-9 epilogue (masking of the scores, output
// normalisation, TMA store).  Every wait is bounded (mbar_wait) and reports
// a code in *err instead of hanging.
//
// Modes: kCausal (outputs + carried state), kState (only the state update
// over a segment, for the two-pass sequence split and the non-causal
// reduction), kApply (non-causal read-out with a fixed global state).
#pragma once

#include "chunk_args.h"
#include "common.cuh"
#include "umma.cuh"

namespace la {
namespace chunk {

using namespace umma;

constexpr int kC = 64;  // tokens per chunk
constexpr int kThreads = 320;
constexpr int kConvWarp0 = 2, kEpiWarp0 = 6;
constexpr int kBarConv = 1, kBarEpi = 2;  // named barriers (0 is __syncthreads)

template <int D, int MODE, bool NORM, bool SPLITK, bool GATED, bool OUT_BF16>
struct Cfg {
    static constexpr bool kHasKV = MODE != kApply;
    static constexpr bool kHasQ = MODE != kState;
    static constexpr int kTile = D * 128;  // 64 rows x D bf16 (D/64 swizzled blocks of 8 KB)
    static constexpr int kZr = D * 16;     // 8 rows x D bf16
    static constexpr int kOutBytes = OUT_BF16 ? 2 : 4;
    // per KV stage: Kb | Kd (gated) | Klo (split) | Vb | Zr | G (256 B, padded)
    static constexpr int kOffKd = kTile;
    static constexpr int kOffKlo = kOffKd + (GATED ? kTile : 0);
    static constexpr int kOffVb = kOffKlo + (SPLITK ? kTile : 0);
    static constexpr int kOffZr = kOffVb + kTile;
    static constexpr int kOffG = kOffZr + (NORM ? kZr : 0);
    static constexpr int kKvStage = kHasKV ? kOffG + 1024 : 0;
    static constexpr int kQStage = kHasQ ? kTile * (GATED ? 2 : 1) : 0;
    static constexpr int kAT = MODE == kCausal ? 2 * 8192 : 0;  // hi + lo, one 64 x 64 block each
    static constexpr int kYStage = kHasQ ? kC * D * kOutBytes : 0;
    static constexpr int kZrApply = MODE == kApply ? kZr : 0;
    static constexpr int kMisc = 4096;  // den, partial Z sums, barriers
    static constexpr int bytes(int nkv, int nq, int ny) {
        return 1024 + nkv * kKvStage + nq * kQStage + 2 * kAT + ny * kYStage + kZrApply + kMisc;
    }
    static constexpr int kLimit = 227 * 1024;
    static constexpr int kNKV = kHasKV ? (bytes(2, kHasQ ? 1 : 0, kHasQ ? 1 : 0) <= kLimit ? 2 : 1) : 0;
    static constexpr int kNY = kHasQ ? (bytes(kNKV, 2, 2) <= kLimit ? 2 : 1) : 0;
    static constexpr int kNQ = kHasQ ? (bytes(kNKV, 2, kNY) <= kLimit ? 2 : 1) : 0;
    static constexpr int kSmem = bytes(kNKV, kNQ, kNY);
    static_assert(kSmem <= kLimit, "shared memory budget");
    // TMEM columns
    static constexpr uint32_t kColS = 0;           // S^T fp32: D columns, lanes = value rows
    static constexpr uint32_t kColHi = D;          // S^T hi bf16 pairs: D/2 columns
    static constexpr uint32_t kColLo = D + D / 2;  // S^T lo
    static constexpr uint32_t kColA = 2 * D;       // two score buffers of 80 columns (64 + 8 for phi(q).Z)
    static constexpr uint32_t kColY = 2 * D + 160; // Y^T: 64 columns
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kColY + 64 <= kTmemCols, "TMEM budget");
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// element (row, k) of a [64 rows][D] K-major swizzled bf16 tile
template <int D>
__device__ __forceinline__ uint32_t tile_off(int row, int k) {
    return static_cast<uint32_t>((k >> 6) * 8192) + sw128_offset(row, (k & 63) * 2);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16& hi, __nv_bfloat16& lo) {
    hi = __float2bfloat16_rn(x);
    lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}
__device__ __forceinline__ __nv_bfloat16& bf_at(uint8_t* base, uint32_t off) {
    return *reinterpret_cast<__nv_bfloat16*>(base + off);
}

template <int D, int MODE, bool NORM, bool SPLITK, bool GATED, bool OUT_BF16>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_kernel(const Args a, const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                 const __grid_constant__ CUtensorMap mapV, const __grid_constant__ CUtensorMap mapY) {
    using Cf = Cfg<D, MODE, NORM, SPLITK, GATED, OUT_BF16>;
    constexpr int NKV = Cf::kNKV, NQ = Cf::kNQ, NY = Cf::kNY;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* kv_base = sm;
    uint8_t* q_base = kv_base + NKV * Cf::kKvStage;
    uint8_t* at_base = q_base + NQ * Cf::kQStage;
    uint8_t* y_base = at_base + 2 * Cf::kAT;
    uint8_t* zr_apply = y_base + NY * Cf::kYStage;
    float* misc = reinterpret_cast<float*>(zr_apply + Cf::kZrApply);
    float* den_s = misc;             // [2][64]
    float* zpart = misc + 128;       // [2][128]
    uint64_t* bars = reinterpret_cast<uint64_t*>(misc + 512);
    uint64_t* full_kv = bars;        // [2]
    uint64_t* empty_kv = bars + 2;   // [2]
    uint64_t* conv_kv = bars + 4;    // [2]
    uint64_t* full_q = bars + 6;     // [2]
    uint64_t* empty_q = bars + 8;    // [2]
    uint64_t* conv_q = bars + 10;    // [2]
    uint64_t* a_full = bars + 12;    // [2]
    uint64_t* a_empty = bars + 14;   // [2]
    uint64_t* at_full = bars + 16;   // [2]
    uint64_t* at_empty = bars + 18;  // [2]
    uint64_t* y_full = bars + 20;
    uint64_t* y_empty = bars + 21;
    uint64_t* state_ready = bars + 22;
    uint64_t* state_done = bars + 23;
    uint64_t* conv_group = bars + 24;  // barrier among the four converter warps
    uint64_t* epi_group = bars + 25;   // barrier among the four epilogue warps
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 26);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x;
    const int seg = blockIdx.y;
    const int b = bh / a.Hkv, hk = bh - b * a.Hkv;
    const int nchunks = (a.T + kC - 1) / kC;
    const int c_begin = seg * a.cps;
    const int nck = min(nchunks, c_begin + a.cps) - c_begin;
    const int G = a.G;

    auto Kb = [&](int s) { return kv_base + s * Cf::kKvStage; };
    auto Kd = [&](int s) { return kv_base + s * Cf::kKvStage + Cf::kOffKd; };
    auto Klo = [&](int s) { return kv_base + s * Cf::kKvStage + Cf::kOffKlo; };
    auto Vb = [&](int s) { return kv_base + s * Cf::kKvStage + Cf::kOffVb; };
    auto Zr = [&](int s) { return MODE == kApply ? zr_apply : kv_base + s * Cf::kKvStage + Cf::kOffZr; };
    auto Gc = [&](int s) { return reinterpret_cast<float*>(kv_base + s * Cf::kKvStage + Cf::kOffG); };
    auto Qb = [&](int s) { return q_base + s * Cf::kQStage; };
    auto Qd = [&](int s) { return q_base + s * Cf::kQStage + Cf::kTile; };
    auto ATh = [&](int s) { return at_base + s * Cf::kAT; };
    auto ATl = [&](int s) { return at_base + s * Cf::kAT + 8192; };
    auto Ys = [&](int s) { return y_base + s * Cf::kYStage; };

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&full_kv[i], 1);
            mbar_init(&empty_kv[i], 1);
            mbar_init(&conv_kv[i], 4);
            mbar_init(&full_q[i], 1);
            mbar_init(&empty_q[i], 1);
            mbar_init(&conv_q[i], 4);
            mbar_init(&a_full[i], 1);
            mbar_init(&a_empty[i], 4);
            mbar_init(&at_full[i], 4);
            mbar_init(&at_empty[i], 1);
        }
        mbar_init(y_full, 1);
        mbar_init(y_empty, 4);
        mbar_init(state_ready, 4);
        mbar_init(state_done, 1);
        mbar_init(conv_group, 4);
        mbar_init(epi_group, 4);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, Cf::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        if (Cf::kHasQ) tma_prefetch(&mapQ);
        if (Cf::kHasKV) {
            tma_prefetch(&mapK);
            tma_prefetch(&mapV);
        }
        if (Cf::kHasQ) tma_prefetch(&mapY);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    unsigned* err = a.err;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            bool ok = true;
            for (int i = 0; i < nck && ok; ++i) {
                const int t0 = (c_begin + i) * kC;
                if (Cf::kHasKV) {
                    const int s = NKV ? i % NKV : 0;
                    if (i >= NKV) ok = mbar_wait(&empty_kv[s], ((i / (NKV ? NKV : 1)) & 1) ^ 1, err, kErrEmptyKV);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&full_kv[s], 2 * Cf::kTile);
                    for (int kb = 0; kb < D / 64; ++kb) {
                        tma_load_4d(Kb(s) + kb * 8192, &mapK, &full_kv[s], kb * 64, hk, t0, b);
                        tma_load_4d(Vb(s) + kb * 8192, &mapV, &full_kv[s], kb * 64, hk, t0, b);
                    }
                }
                if (Cf::kHasQ) {
                    for (int r = 0; r < G && ok; ++r) {
                        const int n = i * G + r, s = n % (NQ ? NQ : 1);
                        if (n >= NQ) ok = mbar_wait(&empty_q[s], ((n / (NQ ? NQ : 1)) & 1) ^ 1, err, kErrEmptyQ);
                        if (!ok) break;
                        mbar_arrive_expect_tx(&full_q[s], Cf::kTile);
                        for (int kb = 0; kb < D / 64; ++kb)
                            tma_load_4d(Qb(s) + kb * 8192, &mapQ, &full_q[s], kb * 64, hk * G + r, t0, b);
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            bool ok = true;
            constexpr uint32_t id_scores = idesc_bf16(64, 64, false, false);
            constexpr uint32_t id_qz = idesc_bf16(64, 8, false, false);
            constexpr uint32_t id_inter = idesc_bf16(D, 64, false, false);
            constexpr uint32_t id_intra = idesc_bf16(D, 64, true, false);
            constexpr uint32_t id_state = idesc_bf16(D, D, true, true);
            const uint32_t tS = tmem + Cf::kColS, tHi = tmem + Cf::kColHi, tLo = tmem + Cf::kColLo;
            const uint32_t tY = tmem + Cf::kColY;
            for (int i = 0; i < nck && ok; ++i) {
                const int s = NKV ? i % NKV : 0;
                if (Cf::kHasKV) {
                    ok = mbar_wait(&conv_kv[s], (i / (NKV ? NKV : 1)) & 1, err, kErrConvKV);
                    if (!ok) break;
                    tc_fence_after();
                }
                if (Cf::kHasQ) {
                    for (int r = 0; r < G && ok; ++r) {
                        const int n = i * G + r, sq = n % (NQ ? NQ : 1), ab = n & 1;
                        ok = mbar_wait(&conv_q[sq], (n / (NQ ? NQ : 1)) & 1, err, kErrConvQ);
                        if (!ok) break;
                        tc_fence_after();
                        uint8_t* qop = GATED ? Qd(sq) : Qb(sq);  // operand of the inter read-out
                        const uint32_t tA = tmem + Cf::kColA + 80 * ab;
                        if (MODE == kCausal || NORM) {
                            if (n >= 2) {
                                ok = mbar_wait(&a_empty[ab], ((n >> 1) & 1) ^ 1, err, kErrAEmpty);
                                if (!ok) break;
                                tc_fence_after();
                            }
                            if (MODE == kCausal) {
                                for (int ks = 0; ks < D / 16; ++ks) {
                                    const uint32_t ko = (ks >> 2) * 8192 + (ks & 3) * 32;
                                    mma_ss(tA, sdesc_sw128(smem_u32(Qb(sq) + ko), 16, 1024),
                                           sdesc_sw128(smem_u32(Kb(s) + ko), 16, 1024), id_scores, ks > 0);
                                }
                            }
                            if (NORM) {
                                for (int ks = 0; ks < D / 16; ++ks) {
                                    const uint32_t ko = (ks >> 2) * 8192 + (ks & 3) * 32;
                                    const uint32_t zo = (ks >> 2) * 1024 + (ks & 3) * 32;
                                    mma_ss(tA + 64, sdesc_sw128(smem_u32(Qb(sq) + ko), 16, 1024),
                                           sdesc_sw128(smem_u32(Zr(s) + zo), 16, 1024), id_qz, ks > 0);
                                }
                            }
                            mma_commit(&a_full[ab]);
                        }
                        if (r == 0 && (MODE == kCausal || i == 0)) {
                            ok = mbar_wait(state_ready, MODE == kCausal ? (i & 1) : 0, err, kErrStateReady);
                            if (!ok) break;
                            tc_fence_after();
                        }
                        if (n >= 1) {
                            ok = mbar_wait(y_empty, (n - 1) & 1, err, kErrYEmpty);
                            if (!ok) break;
                            tc_fence_after();
                        }
                        // inter: Y^T = S_prev^T(hi + lo) . Q^T
                        for (int ks = 0; ks < D / 16; ++ks) {
                            const uint32_t ko = (ks >> 2) * 8192 + (ks & 3) * 32;
                            const uint64_t bq = sdesc_sw128(smem_u32(qop + ko), 16, 1024);
                            mma_ts(tY, tHi + ks * 8, bq, id_inter, ks > 0);
                            mma_ts(tY, tLo + ks * 8, bq, id_inter, 1);
                        }
                        mma_commit(&empty_q[sq]);
                        if (MODE == kCausal) {
                            ok = mbar_wait(&at_full[ab], (n >> 1) & 1, err, kErrATFull);
                            if (!ok) break;
                            tc_fence_after();
                            // intra: Y^T += V^T . A^T (hi + lo)
                            for (int ks = 0; ks < kC / 16; ++ks) {
                                const uint64_t av = sdesc_sw128(smem_u32(Vb(s) + ks * 2048), 8192, 1024);
                                mma_ss(tY, av, sdesc_sw128(smem_u32(ATh(ab) + ks * 32), 16, 1024), id_intra, 1);
                                mma_ss(tY, av, sdesc_sw128(smem_u32(ATl(ab) + ks * 32), 16, 1024), id_intra, 1);
                            }
                            mma_commit(&at_empty[ab]);
                        }
                        mma_commit(y_full);
                    }
                    if (!ok) break;
                }
                if (Cf::kHasKV) {
                    if (MODE == kState && (GATED || i == 0)) {
                        // state mode: the converters publish the (decayed) state before each update
                        ok = mbar_wait(state_ready, i & 1, err, kErrStateReady);
                        if (!ok) break;
                        tc_fence_after();
                    }
                    // state update: S^T += V^T . Kd (+ V^T . Kd_lo)
                    uint8_t* khi = GATED ? Kd(s) : Kb(s);
                    for (int ks = 0; ks < kC / 16; ++ks) {
                        const uint64_t av = sdesc_sw128(smem_u32(Vb(s) + ks * 2048), 8192, 1024);
                        mma_ss(tS, av, sdesc_sw128(smem_u32(khi + ks * 2048), 8192, 1024), id_state, 1);
                        if (SPLITK)
                            mma_ss(tS, av, sdesc_sw128(smem_u32(Klo(s) + ks * 2048), 8192, 1024), id_state, 1);
                    }
                    // the non-gated state pass has no per-chunk hand-off: one phase at the end
                    if (MODE == kCausal || GATED || i == nck - 1) mma_commit(state_done);
                    mma_commit(&empty_kv[s]);
                }
            }
        }
    } else if (warp < kEpiWarp0) {
        // ------------------------------------------------------------ converters
        const int ct = tid - kConvWarp0 * 32;  // 0..127
        const int quad = warp & 3;             // TMEM lane quadrant of this warp
        const int kcol = ct % D;               // feature column handled in tile passes
        const int rgrp = ct / D;               // row group (D = 64: two groups of 32 rows)
        constexpr int kRows = 64 * D / 128;    // rows per thread in tile passes
        const int row0 = rgrp * kRows;
        bool ok = true;
        uint32_t gphase = 0;

        // zero the constant rows 2..7 of every Z-row block
        if (NORM) {
            const int nzr = MODE == kApply ? 1 : NKV;
            for (int z = 0; z < nzr; ++z)
                for (int e = ct; e < D * 8; e += 128) {
                    const int row = e / D, k = e % D;
                    if (row >= 2) bf_at(Zr(z), (k >> 6) * 1024 + sw128_offset(row, (k & 63) * 2)) = __float2bfloat16(0.f);
                }
        }
        // start state -> S^T (fp32) in TMEM; Z in a register of thread k (rgrp 0)
        const float* S_start = nullptr;
        const float* Z_start = nullptr;
        if (MODE == kCausal && a.S_seg) {
            S_start = a.S_seg + ((size_t)bh * a.nseg + seg) * D * D;
            Z_start = a.Z_seg ? a.Z_seg + ((size_t)bh * a.nseg + seg) * D : nullptr;
        } else if (MODE != kState) {
            S_start = a.S_init ? a.S_init + (size_t)bh * D * D : nullptr;
            Z_start = a.Z_init ? a.Z_init + (size_t)bh * D : nullptr;
        }
        // TMEM row of this thread for a D-row accumulator (M = D): value index
        const bool m64 = D == 64;
        const int vrow = m64 ? (quad * 16 + lane) : (quad * 32 + lane);
        const bool vrow_ok = m64 ? lane < 16 : true;
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t r[32];
#pragma unroll
            for (int x = 0; x < 32; ++x)
                r[x] = __float_as_uint((S_start && vrow_ok) ? S_start[(size_t)(c0 + x) * D + vrow] : 0.f);
            tmem_st32(tmem_addr(tmem + Cf::kColS, quad * 32, c0), r);
        }
        tmem_st_wait();
        float zreg = (NORM && Z_start && rgrp == 0) ? Z_start[kcol] : 0.f;
        float gsum = 0.f;  // gated, state mode: total log decay of the segment

        // state hi/lo conversion (and, gated, decay of the fp32 state in place)
        auto convert_state = [&](float decay_mul, bool write_back) {
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(tmem_addr(tmem + Cf::kColS, quad * 32, c0), r);
                tmem_ld_wait();
                reg_fence(r);
                if (MODE != kState) {
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        const float f0 = __uint_as_float(r[2 * x]), f1 = __uint_as_float(r[2 * x + 1]);
                        __nv_bfloat16 h0, l0, h1, l1;
                        split_bf16(f0, h0, l0);
                        split_bf16(f1, h1, l1);
                        __nv_bfloat162 hh, ll;
                        hh.x = h0; hh.y = h1;
                        ll.x = l0; ll.y = l1;
                        hi[x] = *reinterpret_cast<uint32_t*>(&hh);
                        lo[x] = *reinterpret_cast<uint32_t*>(&ll);
                    }
                    tmem_st16(tmem_addr(tmem + Cf::kColHi, quad * 32, c0 / 2), hi);
                    tmem_st16(tmem_addr(tmem + Cf::kColLo, quad * 32, c0 / 2), lo);
                }
                if (write_back) {
#pragma unroll
                    for (int x = 0; x < 32; ++x) r[x] = __float_as_uint(__uint_as_float(r[x]) * decay_mul);
                    tmem_st32(tmem_addr(tmem + Cf::kColS, quad * 32, c0), r);
                }
            }
            tmem_st_wait();
        };

        if (MODE == kApply) {
            // fixed global state: hi/lo once; Z rows from the global key state
            tc_fence_after();
            convert_state(1.f, false);
            if (NORM && rgrp == 0) {
                __nv_bfloat16 h, l;
                split_bf16(zreg, h, l);
                bf_at(Zr(0), (kcol >> 6) * 1024 + sw128_offset(0, (kcol & 63) * 2)) = h;
                bf_at(Zr(0), (kcol >> 6) * 1024 + sw128_offset(1, (kcol & 63) * 2)) = l;
            }
            fence_proxy_async();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(state_ready);
        }

        for (int i = 0; i < nck && ok; ++i) {
            const int t0 = (c_begin + i) * kC;
            const int valid = min(kC, a.T - t0);
            const int s = NKV ? i % NKV : 0;
            float gtot = 0.f;
            if (Cf::kHasKV) {
                ok = warp_wait(&full_kv[s], (i / (NKV ? NKV : 1)) & 1, err, kErrFullKV);
                if (!ok) break;
                float* gc = Gc(s);
                if (GATED) {
                    // inclusive cumulative log decay inside the chunk (first converter warp)
                    if (ct < 32) {
                        float g0 = 0.f, g1 = 0.f;
                        const int j0 = 2 * ct, j1 = 2 * ct + 1;
                        if (j0 < valid) g0 = __bfloat162float(a.decay[((size_t)b * a.T + t0 + j0) * a.Hkv + hk]);
                        if (j1 < valid) g1 = __bfloat162float(a.decay[((size_t)b * a.T + t0 + j1) * a.Hkv + hk]);
                        float sum = g0 + g1, incl = sum;
#pragma unroll
                        for (int o = 1; o < 32; o <<= 1) {
                            const float t = __shfl_up_sync(0xffffffffu, incl, o);
                            if (lane >= o) incl += t;
                        }
                        const float excl = incl - sum;
                        gc[j0] = excl + g0;
                        gc[j1] = excl + sum;
                    }
                    ok = group_sync(conv_group, gphase, err, kErrStateReady);
                    if (!ok) break;
                    gtot = gc[kC - 1];
                }
                // feature map of the keys in place (+ lo part), decayed keys, Z column sums
                float colsum = 0.f;
#pragma unroll 4
                for (int jj = 0; jj < kRows; ++jj) {
                    const int j = row0 + jj;
                    const uint32_t off = tile_off<D>(j, kcol);
                    const float x = __bfloat162float(bf_at(Kb(s), off));
                    if (GATED) {
                        const float w = __expf(gtot - gc[j]);
                        __nv_bfloat16 h, l;
                        split_bf16(x * w, h, l);
                        bf_at(Kd(s), off) = h;
                        bf_at(Klo(s), off) = l;
                    } else {
                        const float f = phi<true>(a.fmap, x, a.eps);
                        if (a.fmap != LA_FMAP_NONE) {
                            __nv_bfloat16 h, l;
                            split_bf16(f, h, l);
                            bf_at(Kb(s), off) = h;
                            if (SPLITK) bf_at(Klo(s), off) = l;
                        } else if (SPLITK) {
                            bf_at(Klo(s), off) = __float2bfloat16(0.f);
                        }
                        if (NORM && j < valid) colsum += f;
                    }
                }
                if (NORM) {
                    // Z rows of this chunk hold Z_prev (hi, lo); then Z += column sums
                    if (D == 128) {
                        __nv_bfloat16 h, l;
                        split_bf16(zreg, h, l);
                        bf_at(Zr(s), (kcol >> 6) * 1024 + sw128_offset(0, (kcol & 63) * 2)) = h;
                        bf_at(Zr(s), (kcol >> 6) * 1024 + sw128_offset(1, (kcol & 63) * 2)) = l;
                        zreg += colsum;
                    } else {
                        zpart[rgrp * 128 + kcol] = colsum;
                        ok = group_sync(conv_group, gphase, err, kErrStateReady);
                        if (!ok) break;
                        if (rgrp == 0) {
                            __nv_bfloat16 h, l;
                            split_bf16(zreg, h, l);
                            bf_at(Zr(s), (kcol >> 6) * 1024 + sw128_offset(0, (kcol & 63) * 2)) = h;
                            bf_at(Zr(s), (kcol >> 6) * 1024 + sw128_offset(1, (kcol & 63) * 2)) = l;
                            zreg += zpart[kcol] + zpart[128 + kcol];
                        }
                        ok = group_sync(conv_group, gphase, err, kErrStateReady);  // zpart reuse
                        if (!ok) break;
                    }
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) mbar_arrive(&conv_kv[s]);
            }
            // state for this chunk, before the query heads (the read-out of head 0
            // needs it, and later heads' loads wait on head 0's read-out):
            // hi/lo of S_prev for the read-out; decay (gated) before the update
            if (MODE == kCausal || (MODE == kState && GATED)) {
                if (i > 0) {
                    ok = warp_wait(state_done, (i - 1) & 1, err, kErrStateDone);
                    if (!ok) break;
                }
                tc_fence_after();
                convert_state(GATED ? __expf(gtot) : 1.f, GATED);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(state_ready);
            } else if (MODE == kState && i == 0) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(state_ready);
            }
            if (Cf::kHasQ) {
                const float* gc = Gc(s);
                for (int r = 0; r < G && ok; ++r) {
                    const int n = i * G + r, sq = n % (NQ ? NQ : 1);
                    ok = warp_wait(&full_q[sq], (n / (NQ ? NQ : 1)) & 1, err, kErrFullQ);
                    if (!ok) break;
                    if (a.fmap != LA_FMAP_NONE || GATED) {
#pragma unroll 4
                        for (int jj = 0; jj < kRows; ++jj) {
                            const int j = row0 + jj;
                            const uint32_t off = tile_off<D>(j, kcol);
                            const float x = __bfloat162float(bf_at(Qb(sq), off));
                            if (GATED) {
                                bf_at(Qd(sq), off) = __float2bfloat16_rn(x * __expf(gc[j]));
                            } else {
                                bf_at(Qb(sq), off) = __float2bfloat16_rn(phi<true>(a.fmap, x, a.eps));
                            }
                        }
                    }
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&conv_q[sq]);
                }
                if (!ok) break;
            }
            if (MODE == kState && GATED) gsum += gtot;
        }

        // final state out: causal (last segment) or every segment in state mode
        const bool write_state = ok && ((MODE == kCausal && seg == a.nseg - 1 && a.S_dst) || MODE == kState);
        if (write_state) {
            // causal: phase nck-1 (one per chunk); non-gated state pass: its single phase
            ok = warp_wait(state_done, (MODE == kState && !GATED) ? 0 : ((nck - 1) & 1), err, kErrStateDone);
            tc_fence_after();
            if (ok) {
                float* Sd = MODE == kState ? a.S_dst + ((size_t)bh * a.nseg + seg) * D * D : a.S_dst + (size_t)bh * D * D;
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tmem_addr(tmem + Cf::kColS, quad * 32, c0), r);
                    tmem_ld_wait();
                    reg_fence(r);
                    if (vrow_ok)
#pragma unroll
                        for (int x = 0; x < 32; ++x) Sd[(size_t)(c0 + x) * D + vrow] = __uint_as_float(r[x]);
                }
                if (NORM && rgrp == 0 && a.Z_dst) {
                    float* Zd = MODE == kState ? a.Z_dst + ((size_t)bh * a.nseg + seg) * D : a.Z_dst + (size_t)bh * D;
                    Zd[kcol] = zreg;
                }
                if (MODE == kState && GATED && ct == 0) a.G_dst[(size_t)bh * a.nseg + seg] = gsum;
            }
        }
    } else {
        // -------------------------------------------------------------- epilogue
        const int et = tid - kEpiWarp0 * 32;  // 0..127
        const int quad = warp & 3;
        const bool m64 = D == 64;
        const int vrow = m64 ? (quad * 16 + lane) : (quad * 32 + lane);  // value index of Y^T row
        const bool vrow_ok = m64 ? lane < 16 : true;
        const int arow = quad * 16 + lane;  // score row (M = 64 layout)
        const bool arow_ok = lane < 16;
        const int n_total = Cf::kHasQ ? nck * G : 0;
        bool ok = true;
        uint32_t gphase = 0;
        for (int n = 0; n <= n_total && ok; ++n) {
            if (n < n_total && (MODE == kCausal || NORM)) {
                // -------- scores of item n: mask, decay, hi/lo split, normaliser
                const int ab = n & 1;
                const int i_chunk = n / G;
                const int s = NKV ? i_chunk % NKV : 0;
                ok = warp_wait(&a_full[ab], (n >> 1) & 1, err, kErrAFull);
                if (!ok) break;
                tc_fence_after();
                const uint32_t tA = tmem + Cf::kColA + 80 * ab;
                uint32_t r[32], r2[32], z[16];
                if (MODE == kCausal) {
                    tmem_ld32(tmem_addr(tA, quad * 32, 0), r);
                    tmem_ld32(tmem_addr(tA, quad * 32, 32), r2);
                }
                if (NORM) tmem_ld16(tmem_addr(tA, quad * 32, 64), z);
                tmem_ld_wait();
                if (MODE == kCausal) {
                    reg_fence(r);
                    reg_fence(r2);
                }
                if (NORM) reg_fence(z);
                float den = 0.f;
                if (NORM) den = __uint_as_float(z[0]) + __uint_as_float(z[1]) + a.eps;
                if (MODE == kCausal) {
                    if (n >= 2) {
                        ok = warp_wait(&at_empty[ab], ((n >> 1) & 1) ^ 1, err, kErrATEmpty);
                        if (!ok) break;
                    }
                    if (arow_ok) {
                        const float* gc = reinterpret_cast<const float*>(Gc(s));
                        const float gi = GATED ? gc[arow] : 0.f;
                        uint8_t* hb = ATh(ab);
                        uint8_t* lb = ATl(ab);
#pragma unroll
                        for (int cch = 0; cch < 8; ++cch) {  // 8 columns per 16-byte chunk
                            uint32_t hv[4], lv[4];
#pragma unroll
                            for (int x = 0; x < 4; ++x) {
                                float v2[2];
#pragma unroll
                                for (int y = 0; y < 2; ++y) {
                                    const int j = cch * 8 + 2 * x + y;
                                    float v = j < 32 ? __uint_as_float(r[j]) : __uint_as_float(r2[j - 32]);
                                    v = (j <= arow) ? v : 0.f;
                                    if (NORM) den += v;
                                    if (GATED && j <= arow) v *= __expf(gi - gc[j]);
                                    v2[y] = v;
                                }
                                __nv_bfloat16 h0, l0, h1, l1;
                                split_bf16(v2[0], h0, l0);
                                split_bf16(v2[1], h1, l1);
                                __nv_bfloat162 hh, ll;
                                hh.x = h0; hh.y = h1;
                                ll.x = l0; ll.y = l1;
                                hv[x] = *reinterpret_cast<uint32_t*>(&hh);
                                lv[x] = *reinterpret_cast<uint32_t*>(&ll);
                            }
                            const uint32_t off = sw128_offset(arow, cch * 16);
                            *reinterpret_cast<uint4*>(hb + off) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                            *reinterpret_cast<uint4*>(lb + off) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
                        }
                    }
                    fence_proxy_async();
                }
                if (NORM && arow_ok) den_s[ab * 64 + arow] = den;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&a_empty[ab]);
                    if (MODE == kCausal) mbar_arrive(&at_full[ab]);
                }
            }
            if (n >= 1) {
                // -------- output of item m = n - 1
                const int m = n - 1;
                const int ab = m & 1;
                const int i_chunk = m / G, r_head = m - i_chunk * G;
                const int t0 = (c_begin + i_chunk) * kC;
                ok = warp_wait(y_full, m & 1, err, kErrYFull);
                if (!ok) break;
                tc_fence_after();
                uint32_t y0[32], y1[32];
                tmem_ld32(tmem_addr(tmem + Cf::kColY, quad * 32, 0), y0);
                tmem_ld32(tmem_addr(tmem + Cf::kColY, quad * 32, 32), y1);
                tmem_ld_wait();
                reg_fence(y0);
                reg_fence(y1);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(y_empty);
                ok = group_sync(epi_group, gphase, err, kErrYFull);  // den_s of item m complete; staging free
                if (!ok) break;
                uint8_t* ys = Ys(m % (NY ? NY : 1));
                if (vrow_ok) {
#pragma unroll
                    for (int x = 0; x < 64; ++x) {
                        float v = x < 32 ? __uint_as_float(y0[x]) : __uint_as_float(y1[x - 32]);
                        if (NORM) v = v / den_s[ab * 64 + x];
                        v *= a.scale;
                        if (OUT_BF16)
                            reinterpret_cast<__nv_bfloat16*>(ys)[x * D + vrow] = __float2bfloat16_rn(v);
                        else
                            reinterpret_cast<float*>(ys)[x * D + vrow] = v;
                    }
                }
                fence_proxy_async();
                ok = group_sync(epi_group, gphase, err, kErrYFull);
                if (!ok) break;
                if (et == 0) {
                    tma_store_4d(&mapY, ys, 0, hk * G + r_head, t0, b);
                    bulk_commit_group();
                    if (NY == 1) bulk_wait_group_read<0>();
                    else bulk_wait_group_read<1>();
                }
            }
        }
        if (et == 0) bulk_wait_group<0>();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cf::kTmemCols);
    }
}

}  // namespace chunk
}  // namespace la
