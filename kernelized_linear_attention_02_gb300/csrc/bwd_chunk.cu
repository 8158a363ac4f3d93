// bwd_chunk.cu -- gradients of the causal linear rule in chunk-parallel form on
// the tensor cores (sm_103a: tcgen05, TMEM, bulk copies), for bf16 inputs with
// Dk = Dv = D in {64, 128}.
//
// "[Feature] LinearAttention layer for Keras", Mathematical definition /
// Causal, with a = phi(q), kt = phi(k) (feature maps of the same request),
// S_t = S0 + sum_{j<=t} kt_j^T v_j, z_t = Z0 + sum_{j<=t} kt_j,
// num_t = a_t S_t, den_t = a_t . z_t + eps (1 without the normalizer) and
// y_t = scale num_t / den_t.  For the incoming gradient dy:
//   ds_t = scale dy_t / den_t,  dd_t = -scale (dy_t . num_t) / den_t^2
//   d a_t  = S_t ds_t + dd_t z_t
//   d kt_j = sum_{t>=j} ((ds_t . v_j) + dd_t) a_t       (over every query head)
//   d v_j  = sum_{t>=j} (a_t . kt_j) ds_t
//   dS0 = sum_t a_t^T ds_t,  dZ0 = sum_t dd_t a_t,  dq = d a o phi'(q), dk = d kt o phi'(k).
// Per chunk c of C = 64 steps with start states S_c, z_c and, from the later
// chunks, R_{c+1} = sum a_t^T ds_t and r_{c+1} = sum dd_t a_t, the sums
// split into a part inside the chunk (masked 64 x 64 products) and a part
// through the states:
//   P   = a kt^T (j <= t),        num = a S_c + P v,   den = a z_c + rowsum(P) + eps
//   Pd  = ds v^T + dd 1^T (j <= t)
//   d a  = ds S_c^T + Pd kt + dd z_c^T
//   d kt = v R_{c+1}^T + 1 r_{c+1}^T + sum_heads Pd^T a
//   d v  = kt R_{c+1}       + sum_heads P^T ds
// Five kernels in stream order:
//   kv     one CTA per chunk: dS_c = kt^T v (tensor cores), dz_c = sum kt
//   scan   forward, element-wise: S_c, z_c of every chunk
//   mid    one CTA per chunk, its query heads one after the other: P, num,
//          den, ds, dd, Pd, d a (-> dq), dR_c = sum a^T ds, dr_c = sum dd a,
//          and the intra parts of d kt and d v
//   scan   reverse, element-wise: R_{c+1}, r_{c+1} of every chunk; dS0, dZ0
//   kvgrad one CTA per chunk: d kt and d v through R_{c+1}, r_{c+1} (-> dk, dv)
// Every fp32 operand of a product enters the tensor cores as bf16 hi + lo
// (about 16 significant bits; the lo x lo product is dropped); the bf16
// inputs (q, k, v, dy) and phi of the identity enter as one part.  Every
// product accumulates in fp32 in TMEM; the scans add in fp32.
#include <algorithm>
#include <atomic>
#include <cstring>

#include "kernels.h"
#include "tiles.cuh"
#include "umma.cuh"

namespace la {
namespace bwd {

using namespace umma;
using namespace tile;

constexpr int kC = 64;
enum : unsigned { kErrLoad = 1u << 20, kErrMma = 1u << 21 };

// Workspace of one chunk (bytes).
template <int D>
struct Lay {
    static constexpr size_t a1k(size_t x) { return (x + 1023) & ~(size_t)1023; }
    static constexpr size_t kDS = 0;                        // fp32 [k][v]: dS_c, then dR_c
    static constexpr size_t kDZ = 4 * D * D;                // fp32 [k]: dz_c, then dr_c
    static constexpr size_t kT = a1k(kDZ + 4 * D);          // S_c, then R_{c+1}: rows v, k contiguous; hi, lo
    static constexpr size_t kV = kT + 4 * D * D;            // fp32 [k]: z_c, then r_{c+1}
    static constexpr size_t kPK = a1k(kV + 4 * D);          // fp32 [j][k]: intra part of d kt
    static constexpr size_t kPV = kPK + 4 * kC * D;         // fp32 [j][v]: intra part of d v
    static constexpr size_t kChunk = kPV + 4 * kC * D;
};

struct BArgs {
    int B, T, Hq, Hkv, G, nc;
    int fmap, norm, out_bf16;
    float eps, scale;
    const __nv_bfloat16 *q, *k, *v, *dy;
    const float *S0, *Z0;
    void *dq, *dk, *dv;
    float *dS0, *dZ0;
    uint8_t* ws;
    unsigned* err;
};

// byte offset of 16-byte chunk cc (8 columns) of row r in a tile of R rows
// stored as 64-column blocks of R x 128 bytes (128-byte swizzle)
template <int R>
__device__ __forceinline__ uint32_t toff(int r, int cc) {
    return (cc >> 3) * (R * 128) + swc(r, cc & 7);
}
template <int R>
__device__ __forceinline__ uint32_t toff_e(int r, int col) {
    return (col >> 6) * (R * 128) + swe(r, col & 63);
}
// K-major operand: R rows (the M or N dimension), K along the columns; step ks of 16 columns
template <int R>
__device__ __forceinline__ uint64_t kdesc(const uint8_t* t, int ks) {
    return sdesc_sw128(smem_u32(t + (ks >> 2) * (R * 128) + (ks & 3) * 32), 16, 1024);
}
// MN-major operand: K along the R rows (step ks of 16 rows), M or N along the columns
template <int R>
__device__ __forceinline__ uint64_t mdesc(const uint8_t* t, int ks) {
    return sdesc_sw128(smem_u32(t + ks * 2048), R * 128, 1024);
}
// TMEM row of an M-row accumulator held by (warp, lane): M = 128 uses every
// lane, M = 64 lanes 0-15 of each quarter (-1: none)
template <int M>
__device__ __forceinline__ int acc_row(int warp, int lane) {
    return M == 128 ? 32 * warp + lane : (lane < 16 ? 16 * warp + lane : -1);
}

__device__ __forceinline__ float phi_f(int fmap, float x, float eps) { return phi<true>(fmap, x, eps); }
// phi' (elu + 1: 1 above zero, e^x below; relu + eps: 1 above zero, 0 below; identity: 1)
__device__ __forceinline__ float dphi_f(int fmap, float x) {
    if (fmap == LA_FMAP_ELU_PLUS_ONE) return x > 0.f ? 1.f : expf(x);
    if (fmap == LA_FMAP_RELU_EPS) return x > 0.f ? 1.f : 0.f;
    return 1.f;
}
// phi' with the fast exponential (about 2 ulp), for the tensor-core path's bar
__device__ __forceinline__ float dphi_fast(int fmap, float x) {
    if (fmap == LA_FMAP_ELU_PLUS_ONE) return x > 0.f ? 1.f : __expf(x);
    if (fmap == LA_FMAP_RELU_EPS) return x > 0.f ? 1.f : 0.f;
    return 1.f;
}
__device__ __forceinline__ void unpack8(uint4 raw, float (&f)[8]) {
    const __nv_bfloat16* p = reinterpret_cast<const __nv_bfloat16*>(&raw);
#pragma unroll
    for (int x = 0; x < 8; ++x) f[x] = __bfloat162float(p[x]);
}

// The 64 token rows (t0 .. t0 + 63, rows at or past nvalid zero) of one head
// of a (B, T, H, D) bf16 tensor, by kNT threads: fetch_rows issues the loads,
// store_rows writes the tile (kMode 0: as they are, 1: phi as one bf16 part,
// 2: phi as hi (tile) and lo (tile + 128 D)); with az, each row's phi (as the
// tile holds it) . z is added into az[row] (shared atomics).  Several
// fetches can be in flight before their stores.
template <int D, int kNT>
struct Rows {
    static constexpr int kCpr = D / 8, kIter = kC * kCpr / kNT;
    uint4 raw[kIter];
};
template <int D, int kNT>
__device__ __forceinline__ void fetch_rows(Rows<D, kNT>& r, const __nv_bfloat16* src, int64_t row0, int64_t rstride,
                                           int nvalid, int tid) {
    constexpr int kCpr = Rows<D, kNT>::kCpr;
#pragma unroll
    for (int i = 0; i < Rows<D, kNT>::kIter; ++i) {
        const int e = tid + kNT * i, t = e / kCpr, cc = e - t * kCpr;
        r.raw[i] = t < nvalid ? *reinterpret_cast<const uint4*>(src + (row0 + t * rstride) * D + 8 * cc)
                              : make_uint4(0, 0, 0, 0);
    }
}
template <int D, int kMode, int kNT>
__device__ __forceinline__ void store_rows(uint8_t* tile, const Rows<D, kNT>& r, int nvalid, int fmap, float eps,
                                           int tid, float* az = nullptr, const float* zc = nullptr) {
    constexpr int kCpr = Rows<D, kNT>::kCpr;
#pragma unroll
    for (int i = 0; i < Rows<D, kNT>::kIter; ++i) {
        const int e = tid + kNT * i, t = e / kCpr, cc = e - t * kCpr;
        const uint32_t off = toff<64>(t, cc);
        if (kMode == 0) {
            st16(tile + off, r.raw[i]);
        } else {
            float f[8];
            unpack8(r.raw[i], f);
#pragma unroll
            for (int x = 0; x < 8; ++x) f[x] = t < nvalid ? phi_f(fmap, f[x], eps) : 0.f;
            uint4 hi, lo;
            split8(f, hi, lo);
            st16(tile + off, hi);
            if (kMode == 2) st16(tile + kC * D * 2 + off, lo);
            if (az && t < nvalid) {
                const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&hi);
                const __nv_bfloat16* l = reinterpret_cast<const __nv_bfloat16*>(&lo);
                float d = 0.f;
#pragma unroll
                for (int x = 0; x < 8; ++x)
                    d = fmaf(__bfloat162float(h[x]) + (kMode == 2 ? __bfloat162float(l[x]) : 0.f), zc[8 * cc + x], d);
                atomicAdd(az + t, d);
            }
        }
    }
}

// x = hi + mid + lo in three bf16 parts (about 24 significant bits), for 8 values
__device__ __forceinline__ void split8x3(const float (&f)[8], uint4& hi, uint4& mid, uint4& lo) {
    float r[8];
    uint32_t* h = &hi.x;
    uint32_t* m = &mid.x;
    uint32_t* l = &lo.x;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        const float2 bf = __bfloat1622float2(b);
        r[2 * i] = f[2 * i] - bf.x;
        r[2 * i + 1] = f[2 * i + 1] - bf.y;
        h[i] = bf2_bits(b);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) split2(r[2 * i], r[2 * i + 1], m[i], l[i]);
}
// sum of the 8 values that hi + lo hold
__device__ __forceinline__ float sum_parts(uint4 hi, uint4 lo) {
    const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&hi);
    const __nv_bfloat16* l = reinterpret_cast<const __nv_bfloat16*>(&lo);
    float s = 0.f;
#pragma unroll
    for (int x = 0; x < 8; ++x) s += __bfloat162float(h[x]) + __bfloat162float(l[x]);
    return s;
}

template <typename TOut>
__device__ __forceinline__ void store8(TOut* p, const float (&f)[8]);
template <>
__device__ __forceinline__ void store8(float* p, const float (&f)[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
}
template <>
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&f)[8]) {
    uint4 hi, lo;
    split8(f, hi, lo);
    *reinterpret_cast<uint4*>(p) = hi;
}

// ------------------------------------------------------------------ kv
template <int D, bool kSplit>
struct KvSmem {
    static constexpr int kK = 0;                   // phi(k): rows j, k contiguous; hi, lo
    static constexpr int kV = 2 * kC * D * 2;      // v: rows j, v contiguous
    static constexpr int kBar = kV + kC * D * 2;
    static constexpr int kBytes = kBar + 64 + 1024;
};

template <int D, bool kSplit>
__global__ void __launch_bounds__(128, 1) bwd_kv_kernel(const __grid_constant__ BArgs a) {
    using L = Lay<D>;
    using S = KvSmem<D, kSplit>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* Kt = sm + S::kK;
    uint8_t* Vt = sm + S::kV;
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + S::kBar);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x / a.nc, c = blockIdx.x - bh * a.nc;
    const int b = bh / a.Hkv, hk = bh - b * a.Hkv;
    const int t0 = c * kC, nvalid = min(kC, a.T - t0);
    uint8_t* wsc = a.ws + ((size_t)bh * a.nc + c) * L::kChunk;

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, D);
        tmem_relinquish();
    }
    const int64_t row0 = ((int64_t)b * a.T + t0) * a.Hkv + hk;
    {
        Rows<D, 128> rk, rv;  // both tiles' loads in flight at once
        fetch_rows<D, 128>(rk, a.k, row0, a.Hkv, nvalid, tid);
        fetch_rows<D, 128>(rv, a.v, row0, a.Hkv, nvalid, tid);
        store_rows<D, kSplit ? 2 : 1, 128>(Kt, rk, nvalid, a.fmap, a.eps, tid);
        store_rows<D, 0, 128>(Vt, rv, nvalid, a.fmap, a.eps, tid);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    if (tid == 0) {
        // dS[k][v] = sum_t kt[t][k] v[t][v]: A = kt (M = k, K = t), B = v (N = v, K = t), both MN-major
        constexpr uint32_t id = idesc_bf16(D, D, true, true);
#pragma unroll
        for (int ks = 0; ks < kC / 16; ++ks) {
            mma_ss(tmem, mdesc<64>(Kt, ks), mdesc<64>(Vt, ks), id, ks > 0);
            if (kSplit) mma_ss(tmem, mdesc<64>(Kt + kC * D * 2, ks), mdesc<64>(Vt, ks), id, 1);
        }
        mma_commit(bar);
    }
    // dz[k] = sum_t phi(k[t][k]) in fp32 while the product runs, from the key
    // tile itself: phi as the products see it (hi + lo, or one part), so that z
    // and S describe the same keys; rows past the sequence hold zeros
    if (a.norm && tid < D) {
        float z = 0.f;
#pragma unroll 8
        for (int t = 0; t < kC; ++t) {
            const uint32_t off = toff_e<64>(t, tid);
            float f = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(Kt + off));
            if (kSplit) f += __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(Kt + kC * D * 2 + off));
            z += f;
        }
        reinterpret_cast<float*>(wsc + L::kDZ)[tid] = z;
    }
    const bool ok = __syncthreads_and(warp_wait(bar, 0, a.err, kErrMma));
    tc_fence_after();
    if (ok) {
        const int row = acc_row<D>(warp, lane);
        float* ds = reinterpret_cast<float*>(wsc + L::kDS);
#pragma unroll 1
        for (int c32 = 0; c32 < D / 32; ++c32) {
            uint32_t r[32];
            tmem_ld32(tmem_addr(tmem, 32 * warp, 32 * c32), r);
            tmem_ld_wait();
            reg_fence(r);
            if (row >= 0) {
                float4* dst = reinterpret_cast<float4*>(ds + (size_t)row * D + 32 * c32);
#pragma unroll
                for (int x = 0; x < 8; ++x)
                    dst[x] = make_float4(__uint_as_float(r[4 * x]), __uint_as_float(r[4 * x + 1]),
                                         __uint_as_float(r[4 * x + 2]), __uint_as_float(r[4 * x + 3]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, D);
    }
}

// ------------------------------------------------------------------ scan
// The chunk states as prefix sums over the chunks, element by element:
// forward, S_c = S0 + sum_{c'<c} dS_c' and z_c; reverse, R_{c+1} =
// sum_{c'>c} dR_c' and r_{c+1}, then dS0 = R_0 and dZ0 = r_0.  Each chunk's
// matrix goes to its tile (rows v, k contiguous, hi and lo) and its vector to
// kV.  A CTA owns 32 values v of one key group of 4 (and, for key group 0,
// the vector elements v) and splits the chunks into kScanSegs segments, one
// warp each: pass 1 sums each segment's increments (independent loads, all in
// flight), the segments' offsets follow from those sums in shared memory,
// and pass 2 walks each segment again writing the running state, so no thread
// walks more than nc / kScanSegs chunks in sequence.
constexpr int kScanThreads = 256;
constexpr int kScanRows = 4;
constexpr int kScanSegs = kScanThreads / 32;
template <int D>
constexpr int scan_ctas() { return D * D / kScanRows / 32; }

template <int D, bool kRev>
__global__ void __launch_bounds__(kScanThreads) bwd_scan_kernel(const __grid_constant__ BArgs a) {
    using L = Lay<D>;
    constexpr int kCtas = scan_ctas<D>();
    constexpr int R = kScanRows;
    __shared__ float part[kScanSegs][32][R + 1];
    const int bh = blockIdx.x / kCtas;
    const int e = blockIdx.x - bh * kCtas;           // element block: 32 values v x one key group
    const int lane = threadIdx.x & 31, seg = threadIdx.x >> 5;
    const int v = 32 * (e % (D / 32)) + lane, k0 = R * (e / (D / 32));
    const bool vec = a.norm && k0 == 0;  // also carries vector element v
    const int nc = a.nc;
    uint8_t* ws0 = a.ws + (size_t)bh * nc * L::kChunk;
    // 8-byte half of the 16-byte chunk that holds keys k0 .. k0 + 3 of row v
    const uint32_t soff = (k0 >> 6) * (D * 128) + swc(v, (k0 & 63) >> 3) + ((k0 & 4) ? 8 : 0);
    // this warp's segment of the walk order (reverse: chunks nc-1 .. 0)
    const int per = (nc + kScanSegs - 1) / kScanSegs;
    const int i0 = min(nc, seg * per), i1 = min(nc, i0 + per);
    auto chunk_of = [&](int i) { return kRev ? nc - 1 - i : i; };
    auto load = [&](int i, float (&n)[R], float& x) {
        const uint8_t* w = ws0 + (size_t)chunk_of(i) * L::kChunk;
        const float* d = reinterpret_cast<const float*>(w + L::kDS);
#pragma unroll
        for (int q = 0; q < R; ++q) n[q] = d[(k0 + q) * D + v];
        x = vec ? reinterpret_cast<const float*>(w + L::kDZ)[v] : 0.f;
    };

    // pass 1: this segment's sum, eight chunks of loads at a time
    float tot[R] = {0.f, 0.f, 0.f, 0.f}, totv = 0.f;
#pragma unroll 1
    for (int i = i0; i < i1; i += 8) {
        float n8[8][R], x8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (i + u < i1) {
                load(i + u, n8[u], x8[u]);
            } else {
#pragma unroll
                for (int q = 0; q < R; ++q) n8[u][q] = 0.f;
                x8[u] = 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
#pragma unroll
            for (int q = 0; q < R; ++q) tot[q] += n8[u][q];
            totv += x8[u];
        }
    }
#pragma unroll
    for (int q = 0; q < R; ++q) part[seg][lane][q] = tot[q];
    part[seg][lane][R] = totv;
    __syncthreads();

    // the state entering this segment: the start value plus the earlier segments' sums
    float m[R], mv = 0.f;
#pragma unroll
    for (int q = 0; q < R; ++q) m[q] = (!kRev && a.S0) ? a.S0[(size_t)bh * D * D + (size_t)(k0 + q) * D + v] : 0.f;
    if (!kRev && vec && a.Z0) mv = a.Z0[(size_t)bh * D + v];
    for (int sg = 0; sg < seg; ++sg) {
#pragma unroll
        for (int q = 0; q < R; ++q) m[q] += part[sg][lane][q];
        mv += part[sg][lane][R];
    }

    // pass 2: the running state of every chunk of the segment
#pragma unroll 1
    for (int i = i0; i < i1; i += 8) {
        float n8[8][R], x8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (i + u < i1) load(i + u, n8[u], x8[u]);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (i + u < i1) {
                uint8_t* w = ws0 + (size_t)chunk_of(i + u) * L::kChunk;
                uint32_t hi[R / 2], lo[R / 2];
#pragma unroll
                for (int x = 0; x < R / 2; ++x) split2(m[2 * x], m[2 * x + 1], hi[x], lo[x]);
                *reinterpret_cast<uint2*>(w + L::kT + soff) = make_uint2(hi[0], hi[1]);
                *reinterpret_cast<uint2*>(w + L::kT + 2 * D * D + soff) = make_uint2(lo[0], lo[1]);
                if (vec) reinterpret_cast<float*>(w + L::kV)[v] = mv;
#pragma unroll
                for (int q = 0; q < R; ++q) m[q] += n8[u][q];
                mv += x8[u];
            }
        }
    }
    // reverse: after the last segment, the total is dS0 (and dZ0)
    if (kRev && seg == kScanSegs - 1) {
        if (a.dS0) {
#pragma unroll
            for (int q = 0; q < R; ++q) a.dS0[(size_t)bh * D * D + (size_t)(k0 + q) * D + v] = m[q];
        }
        if (vec && a.dZ0) a.dZ0[(size_t)bh * D + v] = mv;
    }
}

// ------------------------------------------------------------------ mid
template <int D>
struct MidSmem {
    static constexpr int kTok = kC * D * 2;       // one bf16 part of a 64-row tile of D columns
    static constexpr int kPart = kC * kC * 2;     // one bf16 part of the 64 x 64 weights
    static constexpr int kK = 0;                  // phi(k): rows j; hi, lo
    static constexpr int kV = kK + 2 * kTok;      // v: rows j
    static constexpr int kS = kV + kTok;          // S_c: rows v, k contiguous; hi, lo
    static constexpr int kQ = kS + 4 * D * D;     // phi(q) of the head: rows t; hi, lo
    static constexpr int kY = kQ + 2 * kTok;      // dy of the head: rows t
    static constexpr int kP = kY + kTok;          // P, then Pd: rows t, j contiguous; hi, mid, lo
    static constexpr int kDs = kP + 3 * kPart;    // ds: rows t, v contiguous; hi, mid
    static constexpr int kF = kDs + 2 * kTok;     // fp32: z_c [D], den, dd, phi(q) . z_c [64 each], half sums [2][64] x 2
    static constexpr int kBar = kF + 4 * (D + 448);
    static constexpr int kBytes = kBar + 64 + 1024;
};
// TMEM columns: token-row products (a)-(d) share kTokAcc (D columns); dR,
// the intra d v^T and the intra d kt^T accumulate over the query heads.  256
// columns at D = 64, so two CTAs share an SM.
template <int D>
struct MidTmem {
    static constexpr uint32_t kTokAcc = 0, kR = D, kF = 2 * D, kG = 2 * D + 64;
    static constexpr uint32_t kCols = D == 64 ? 256 : 512;
};

template <int D, bool kSplit>
__global__ void __launch_bounds__(256, D == 64 ? 2 : 1) bwd_mid_kernel(const __grid_constant__ BArgs a) {
    using L = Lay<D>;
    using S = MidSmem<D>;
    using TM = MidTmem<D>;
    constexpr int kTok = S::kTok, kPart = S::kPart;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* Kt = sm + S::kK;
    uint8_t* Vt = sm + S::kV;
    uint8_t* St = sm + S::kS;
    uint8_t* Qt = sm + S::kQ;
    uint8_t* Yt = sm + S::kY;
    uint8_t* Pt = sm + S::kP;
    uint8_t* Dt = sm + S::kDs;
    float* zc = reinterpret_cast<float*>(sm + S::kF);
    float* den_s = zc + D;
    float* dd_s = den_s + 64;
    float* az = dd_s + 64;
    float* rsp = az + 64;      // [2][64] row sums of P over each column half
    float* dotp = rsp + 128;   // [2][64] dy . num over each column half
    uint64_t* bar_ld = reinterpret_cast<uint64_t*>(sm + S::kBar);
    uint64_t* bar_mma = bar_ld + 1;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bar_ld + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x / a.nc, c = blockIdx.x - bh * a.nc;
    const int b = bh / a.Hkv, hk = bh - b * a.Hkv;
    const int t0 = c * kC, nvalid = min(kC, a.T - t0), G = a.G;
    const bool norm = a.norm != 0;
    uint8_t* wsc = a.ws + ((size_t)bh * a.nc + c) * L::kChunk;
    unsigned* err = a.err;

    if (tid == 0) {
        mbar_init(bar_ld, 1);
        mbar_init(bar_mma, 1);
        fence_barrier_init();
        mbar_arrive_expect_tx(bar_ld, 4 * D * D);
        bulk_load(St, wsc + L::kT, 4 * D * D, bar_ld);
    }
    if (warp == 0) {
        tmem_alloc(tslot, TM::kCols);
        tmem_relinquish();
    }
    const int64_t krow0 = ((int64_t)b * a.T + t0) * a.Hkv + hk;
    const int64_t qrow00 = ((int64_t)b * a.T + t0) * a.Hq + (int64_t)hk * G;  // first query head's rows
    {
        // keys, values and the first head's queries and dy: every load in flight at once
        Rows<D, 256> rk, rv, rq, ry;
        fetch_rows<D, 256>(rk, a.k, krow0, a.Hkv, nvalid, tid);
        fetch_rows<D, 256>(rv, a.v, krow0, a.Hkv, nvalid, tid);
        fetch_rows<D, 256>(rq, a.q, qrow00, a.Hq, nvalid, tid);
        fetch_rows<D, 256>(ry, a.dy, qrow00, a.Hq, nvalid, tid);
        if (tid < D) zc[tid] = norm ? reinterpret_cast<const float*>(wsc + L::kV)[tid] : 0.f;
        if (tid < 64) az[tid] = 0.f;
        __syncthreads();  // z_c and the zeroed row sums before the query tile's dot products
        store_rows<D, kSplit ? 2 : 1, 256>(Kt, rk, nvalid, a.fmap, a.eps, tid);
        store_rows<D, 0, 256>(Vt, rv, nvalid, a.fmap, a.eps, tid);
        store_rows<D, kSplit ? 2 : 1, 256>(Qt, rq, nvalid, a.fmap, a.eps, tid, norm ? az : nullptr, zc);
        store_rows<D, 0, 256>(Yt, ry, nvalid, a.fmap, a.eps, tid);
    }
    bool ok = warp_wait(bar_ld, 0, err, kErrLoad);
    tc_fence_before();
    ok = __syncthreads_and(ok);
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tTok = tmem + TM::kTokAcc;

    constexpr uint32_t idA = idesc_bf16(64, 64, false, false);  // P = a kt^T
    constexpr uint32_t idQS = idesc_bf16(64, D, false, false);  // a S_c: B = S^T rows v, K = k
    constexpr uint32_t idPV = idesc_bf16(64, D, false, true);   // P v: B = v MN-major
    constexpr uint32_t idDV = idesc_bf16(64, 64, false, false); // ds v^T: B = v rows j, K = v
    constexpr uint32_t idR = idesc_bf16(D, D, true, true);      // a^T ds
    constexpr uint32_t idF = idesc_bf16(D, 64, true, true);     // ds^T P and a^T Pd
    constexpr uint32_t idDS = idesc_bf16(64, D, false, true);   // ds S_c^T and Pd kt: B MN-major
    uint32_t ph = 0;
    // Epilogues: warps w and w + 4 read the same TMEM lane quarter (w); warp w
    // takes the first half of the columns, warp w + 4 the second.  Token-row
    // products (M = 64) live in lanes 0-15 of each quarter.
    const int quarter = warp & 3, half = warp >> 2;
    const int trow = 16 * quarter + (lane & 15);  // token row of this thread (lanes 0-15)
    const bool has_row = lane < 16;
    float racc = 0.f;  // dr_c[tid] over the heads

    auto mma_round = [&](auto&& issue) -> bool {  // one batch of products, block-uniform result
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            issue();
            mma_commit(bar_mma);
        }
        bool w = warp_wait(bar_mma, ph++ & 1, err, kErrMma);
        w = __syncthreads_and(w);
        tc_fence_after();
        return w;
    };

#pragma unroll 1
    for (int r = 0; r < G && ok; ++r) {
        const int hq = hk * G + r;
        const int64_t qrow0 = ((int64_t)b * a.T + t0) * a.Hq + hq;
        if (r > 0) {  // (the first head's rows were loaded with the keys)
            Rows<D, 256> rq, ry;
            fetch_rows<D, 256>(rq, a.q, qrow0, a.Hq, nvalid, tid);
            fetch_rows<D, 256>(ry, a.dy, qrow0, a.Hq, nvalid, tid);
            store_rows<D, kSplit ? 2 : 1, 256>(Qt, rq, nvalid, a.fmap, a.eps, tid, norm ? az : nullptr, zc);
            store_rows<D, 0, 256>(Yt, ry, nvalid, a.fmap, a.eps, tid);
        }

        // (a) P = a kt^T and a . z_c
        ok = mma_round([&] {
#pragma unroll 1
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint64_t qh = kdesc<64>(Qt, ks), kh = kdesc<64>(Kt, ks);
                mma_ss(tTok, qh, kh, idA, ks > 0);
                if (kSplit) {  // all four products: P is (a_hi + a_lo) . (kt_hi + kt_lo) to fp32 rounding
                    const uint64_t ql = kdesc<64>(Qt + kTok, ks), kl = kdesc<64>(Kt + kTok, ks);
                    mma_ss(tTok, qh, kl, idA, 1);
                    mma_ss(tTok, ql, kh, idA, 1);
                    mma_ss(tTok, ql, kl, idA, 1);
                }
            }
        });
        if (!ok) break;
        {
            // P row (this half's 32 columns) in three parts, and its row sum
            uint32_t r0[32];
            tmem_ld32(tmem_addr(tTok, 32 * quarter, 32 * half), r0);
            tmem_ld_wait();
            reg_fence(r0);
            if (has_row) {
                const bool tv = trow < nvalid;
                float rs = 0.f;
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const int cc = 4 * half + c4;
                    float f8[8];
#pragma unroll
                    for (int x = 0; x < 8; ++x) {
                        const int j = 8 * cc + x;
                        f8[x] = (tv && j <= trow) ? __uint_as_float(r0[8 * c4 + x]) : 0.f;
                    }
                    uint4 hi, mid, lo;
                    split8x3(f8, hi, mid, lo);
                    st16(Pt + toff<64>(trow, cc), hi);
                    st16(Pt + kPart + toff<64>(trow, cc), mid);
                    st16(Pt + 2 * kPart + toff<64>(trow, cc), lo);
                    // the weights exactly as the product P v sees them, so that
                    // y = num / den is the weighted mean the gradient's sums assume
                    rs += sum_parts(hi, mid) + sum_parts(lo, make_uint4(0, 0, 0, 0));
                }
                rsp[64 * half + trow] = rs;
            }
        }
        // (b) num = a S_c + P v
        ok = mma_round([&] {
#pragma unroll 1
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint64_t qh = kdesc<64>(Qt, ks), sh = kdesc<D>(St, ks);
                mma_ss(tTok, qh, sh, idQS, ks > 0);
                const uint64_t sl = kdesc<D>(St + 2 * D * D, ks);
                mma_ss(tTok, qh, sl, idQS, 1);
                if (kSplit) {
                    const uint64_t ql = kdesc<64>(Qt + kTok, ks);
                    mma_ss(tTok, ql, sh, idQS, 1);
                    mma_ss(tTok, ql, sl, idQS, 1);
                }
            }
#pragma unroll 1
            for (int ks = 0; ks < kC / 16; ++ks) {
                const uint64_t bv = mdesc<64>(Vt, ks);
#pragma unroll
                for (int part = 0; part < 3; ++part) mma_ss(tTok, kdesc<64>(Pt + part * kPart, ks), bv, idPV, 1);
            }
        });
        if (!ok) break;
        {
            // ds = scale dy / den in three bf16 parts (hi and mid in Dt, lo over
            // dy's own row of Yt once it is read), dd = -scale (dy . num) / den^2
            const float den =
                has_row ? (norm ? rsp[trow] + rsp[64 + trow] + az[trow] + a.eps : 1.f) : 1.f;
            if (has_row && half == 0) den_s[trow] = den;
            const float sden = a.scale / den;
            const bool tv = has_row && trow < nvalid;
            float dot = 0.f;
#pragma unroll 1
            for (int c32 = 0; c32 < D / 64; ++c32) {
                const int col = (D / 2) * half + 32 * c32;
                uint32_t rn[32];
                tmem_ld32(tmem_addr(tTok, 32 * quarter, col), rn);
                tmem_ld_wait();
                reg_fence(rn);
                if (has_row) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int cc = col / 8 + q4;
                        float dyv[8], dsv[8];
                        unpack8(*reinterpret_cast<const uint4*>(Yt + toff<64>(trow, cc)), dyv);
#pragma unroll
                        for (int x = 0; x < 8; ++x) {
                            dot = fmaf(dyv[x], __uint_as_float(rn[8 * q4 + x]), dot);
                            dsv[x] = tv ? sden * dyv[x] : 0.f;
                        }
                        uint4 hi, mid, lo;
                        split8x3(dsv, hi, mid, lo);
                        st16(Dt + toff<64>(trow, cc), hi);
                        st16(Dt + kTok + toff<64>(trow, cc), mid);
                        st16(Yt + toff<64>(trow, cc), lo);
                    }
                }
            }
            if (has_row) dotp[64 * half + trow] = dot;
        }
        // (c) ds v^T (all three parts of ds: Pd = ds v^T + dd cancels to
        // nearly zero where y_t is close to v_j); (e) dR += a^T ds; (f) d v^T += ds^T P
        ok = mma_round([&] {
#pragma unroll 1
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint64_t bv = kdesc<64>(Vt, ks);
                mma_ss(tTok, kdesc<64>(Dt, ks), bv, idDV, ks > 0);
                mma_ss(tTok, kdesc<64>(Dt + kTok, ks), bv, idDV, 1);
                mma_ss(tTok, kdesc<64>(Yt, ks), bv, idDV, 1);
            }
#pragma unroll 1
            for (int ks = 0; ks < kC / 16; ++ks) {
                const uint32_t acc = (r > 0 || ks > 0) ? 1u : 0u;
                const uint64_t qh = mdesc<64>(Qt, ks), dh = mdesc<64>(Dt, ks), dl = mdesc<64>(Dt + kTok, ks);
                const uint64_t ph_ = mdesc<64>(Pt, ks), pl = mdesc<64>(Pt + kPart, ks);
                mma_ss(tmem + TM::kR, qh, dh, idR, acc);
                mma_ss(tmem + TM::kR, qh, dl, idR, 1);
                if (kSplit) mma_ss(tmem + TM::kR, mdesc<64>(Qt + kTok, ks), dh, idR, 1);
                mma_ss(tmem + TM::kF, dh, ph_, idF, acc);
                mma_ss(tmem + TM::kF, dh, pl, idF, 1);
                mma_ss(tmem + TM::kF, dl, ph_, idF, 1);
            }
        });
        if (!ok) break;
        {
            // Pd = ds v^T + dd (j <= t), dd = -scale (dy . num) / den^2
            uint32_t r0[32];
            tmem_ld32(tmem_addr(tTok, 32 * quarter, 32 * half), r0);
            tmem_ld_wait();
            reg_fence(r0);
            if (has_row) {
                const bool tv = trow < nvalid;
                const float den = den_s[trow];
                const float dd = (tv && norm) ? -a.scale * (dotp[trow] + dotp[64 + trow]) / (den * den) : 0.f;
                if (half == 0) {
                    dd_s[trow] = dd;
                    az[trow] = 0.f;  // for the next head (its loader runs after two barriers)
                }
                // three parts: Pd kt sums terms that cancel (a query with few active
                // feature dimensions has d a ~ 0 along them)
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const int cc = 4 * half + c4;
                    float f8[8];
#pragma unroll
                    for (int x = 0; x < 8; ++x) {
                        const int j = 8 * cc + x;
                        f8[x] = (tv && j <= trow) ? __uint_as_float(r0[8 * c4 + x]) + dd : 0.f;
                    }
                    uint4 hi, mid, lo;
                    split8x3(f8, hi, mid, lo);
                    st16(Pt + toff<64>(trow, cc), hi);
                    st16(Pt + kPart + toff<64>(trow, cc), mid);
                    st16(Pt + 2 * kPart + toff<64>(trow, cc), lo);
                }
            }
        }
        // (d) d a = ds S_c^T + Pd kt; (g) d kt^T += a^T Pd
        ok = mma_round([&] {
#pragma unroll 1
            for (int ks = 0; ks < D / 16; ++ks) {
                // ds (three parts) against S_c (hi + lo): every product above 2^-24 of the largest
                const uint64_t d0 = kdesc<64>(Dt, ks), d1 = kdesc<64>(Dt + kTok, ks), d2 = kdesc<64>(Yt, ks);
                const uint64_t sh = mdesc<D>(St, ks), sl = mdesc<D>(St + 2 * D * D, ks);
                mma_ss(tTok, d0, sh, idDS, ks > 0);
                mma_ss(tTok, d0, sl, idDS, 1);
                mma_ss(tTok, d1, sh, idDS, 1);
                mma_ss(tTok, d1, sl, idDS, 1);
                mma_ss(tTok, d2, sh, idDS, 1);
            }
#pragma unroll 1
            for (int ks = 0; ks < kC / 16; ++ks) {
                const uint32_t acc = (r > 0 || ks > 0) ? 1u : 0u;
                const uint64_t kh = mdesc<64>(Kt, ks);
#pragma unroll
                for (int part = 0; part < 3; ++part) mma_ss(tTok, kdesc<64>(Pt + part * kPart, ks), kh, idDS, 1);
                if (kSplit) {
                    const uint64_t kl = mdesc<64>(Kt + kTok, ks);
                    mma_ss(tTok, kdesc<64>(Pt, ks), kl, idDS, 1);
                    mma_ss(tTok, kdesc<64>(Pt + kPart, ks), kl, idDS, 1);
                }
                const uint64_t qh = mdesc<64>(Qt, ks), bph = mdesc<64>(Pt, ks), bpl = mdesc<64>(Pt + kPart, ks);
                mma_ss(tmem + TM::kG, qh, bph, idF, acc);
                mma_ss(tmem + TM::kG, qh, bpl, idF, 1);
                if (kSplit) mma_ss(tmem + TM::kG, mdesc<64>(Qt + kTok, ks), bph, idF, 1);
            }
        });
        if (!ok) break;
        {
            // dq = (d a + dd z_c) o phi'(q)
            const bool tv = has_row && trow < nvalid;
            const float dd = has_row ? dd_s[trow] : 0.f;
            const __nv_bfloat16* qr = a.q + (qrow0 + (int64_t)(tv ? trow : 0) * a.Hq) * D;
#pragma unroll 1
            for (int c32 = 0; c32 < D / 64; ++c32) {
                const int col = (D / 2) * half + 32 * c32;
                uint32_t rd[32];
                tmem_ld32(tmem_addr(tTok, 32 * quarter, col), rd);
                tmem_ld_wait();
                reg_fence(rd);
                if (tv) {
                    uint4 qraw[4];
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) qraw[q4] = *reinterpret_cast<const uint4*>(qr + col + 8 * q4);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int k0 = col + 8 * q4;
                        float qx[8], o[8];
                        unpack8(qraw[q4], qx);
#pragma unroll
                        for (int x = 0; x < 8; ++x)
                            o[x] = (__uint_as_float(rd[8 * q4 + x]) + (norm ? dd * zc[k0 + x] : 0.f)) *
                                   dphi_f(a.fmap, qx[x]);
                        const int64_t o0 = (qrow0 + (int64_t)trow * a.Hq) * D + k0;
                        if (a.out_bf16)
                            store8(static_cast<__nv_bfloat16*>(a.dq) + o0, o);
                        else
                            store8(static_cast<float*>(a.dq) + o0, o);
                    }
                }
            }
            // dr_c[k] += sum_t phi(q)[t][k] dd_t (k = tid)
            if (norm && tid < D) {
                float s = 0.f;
#pragma unroll 8
                for (int t = 0; t < nvalid; ++t) {
                    const uint32_t off = toff_e<64>(t, tid);
                    float x = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(Qt + off));
                    if (kSplit) x += __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(Qt + kTok + off));
                    s = fmaf(x, dd_s[t], s);
                }
                racc += s;
            }
        }
        tc_fence_before();
        __syncthreads();  // Qt, Yt, Pt, Dt and the token accumulator are free for the next head
        tc_fence_after();
    }
    if (ok) {
        // dR_c -> kDS ([k][v]), dr_c -> kDZ, intra d v -> kPV ([j][v]), intra d kt -> kPK ([j][k])
        const int row = acc_row<D>(quarter, lane);
        float* dR = reinterpret_cast<float*>(wsc + L::kDS);
#pragma unroll 1
        for (int c32 = 0; c32 < D / 64; ++c32) {
            const int col = (D / 2) * half + 32 * c32;
            uint32_t rr[32];
            tmem_ld32(tmem_addr(tmem + TM::kR, 32 * quarter, col), rr);
            tmem_ld_wait();
            reg_fence(rr);
            if (row >= 0) {
                float4* dst = reinterpret_cast<float4*>(dR + (size_t)row * D + col);
#pragma unroll
                for (int x = 0; x < 8; ++x)
                    dst[x] = make_float4(__uint_as_float(rr[4 * x]), __uint_as_float(rr[4 * x + 1]),
                                         __uint_as_float(rr[4 * x + 2]), __uint_as_float(rr[4 * x + 3]));
            }
        }
        float* pv = reinterpret_cast<float*>(wsc + L::kPV);
        float* pk = reinterpret_cast<float*>(wsc + L::kPK);
        {
            const int h = half;
            uint32_t rf[32], rg[32];
            tmem_ld32(tmem_addr(tmem + TM::kF, 32 * quarter, 32 * h), rf);
            tmem_ld32(tmem_addr(tmem + TM::kG, 32 * quarter, 32 * h), rg);
            tmem_ld_wait();
            reg_fence(rf);
            reg_fence(rg);
            if (row >= 0) {
#pragma unroll
                for (int x = 0; x < 32; ++x) {
                    pv[(32 * h + x) * D + row] = __uint_as_float(rf[x]);
                    pk[(32 * h + x) * D + row] = __uint_as_float(rg[x]);
                }
            }
        }
        if (norm && tid < D) reinterpret_cast<float*>(wsc + L::kDZ)[tid] = racc;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TM::kCols);
    }
}

// ------------------------------------------------------------------ kvgrad
template <int D>
struct KgSmem {
    static constexpr int kR = 0;                  // R_{c+1}: rows v, k contiguous; hi, lo
    static constexpr int kK = 4 * D * D;          // phi(k): rows j; hi, lo
    static constexpr int kV = kK + 2 * kC * D * 2;  // v: rows j
    static constexpr int kF = kV + kC * D * 2;    // r_{c+1} [D]
    static constexpr int kBar = kF + 4 * D;
    static constexpr int kBytes = kBar + 64 + 1024;
};

template <int D, bool kSplit>
__global__ void __launch_bounds__(256, 1) bwd_kvgrad_kernel(const __grid_constant__ BArgs a) {
    using L = Lay<D>;
    using S = KgSmem<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* Rt = sm + S::kR;
    uint8_t* Kt = sm + S::kK;
    uint8_t* Vt = sm + S::kV;
    float* rv = reinterpret_cast<float*>(sm + S::kF);
    uint64_t* bar_ld = reinterpret_cast<uint64_t*>(sm + S::kBar);
    uint64_t* bar_mma = bar_ld + 1;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bar_ld + 2);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x / a.nc, c = blockIdx.x - bh * a.nc;
    const int b = bh / a.Hkv, hk = bh - b * a.Hkv;
    const int t0 = c * kC, nvalid = min(kC, a.T - t0);
    const uint8_t* wsc = a.ws + ((size_t)bh * a.nc + c) * L::kChunk;

    if (tid == 0) {
        mbar_init(bar_ld, 1);
        mbar_init(bar_mma, 1);
        fence_barrier_init();
        mbar_arrive_expect_tx(bar_ld, 4 * D * D);
        bulk_load(Rt, wsc + L::kT, 4 * D * D, bar_ld);
    }
    if (warp == 0) {
        tmem_alloc(tslot, 2 * D);
        tmem_relinquish();
    }
    const int64_t row0 = ((int64_t)b * a.T + t0) * a.Hkv + hk;
    {
        Rows<D, 256> rk, rv;  // both tiles' loads in flight at once
        fetch_rows<D, 256>(rk, a.k, row0, a.Hkv, nvalid, tid);
        fetch_rows<D, 256>(rv, a.v, row0, a.Hkv, nvalid, tid);
        store_rows<D, kSplit ? 2 : 1, 256>(Kt, rk, nvalid, a.fmap, a.eps, tid);
        store_rows<D, 0, 256>(Vt, rv, nvalid, a.fmap, a.eps, tid);
    }
    if (tid < D) rv[tid] = a.norm ? reinterpret_cast<const float*>(wsc + L::kV)[tid] : 0.f;
    bool ok = warp_wait(bar_ld, 0, a.err, kErrLoad);
    fence_proxy_async();
    tc_fence_before();
    ok = __syncthreads_and(ok);
    tc_fence_after();
    const uint32_t tmem = *tslot;
    if (ok) {
        if (tid == 0) {
            // token-row products (rows j, M = 64):
            //   d kt = v R^T:  A = v (rows j, K = v), B = R as (N = k, K = v): MN-major
            //   d v  = kt R:   A = kt (rows j, K = k), B = R^T as (N = v, K = k): K-major
            constexpr uint32_t idK = idesc_bf16(64, D, false, true);
            constexpr uint32_t idV = idesc_bf16(64, D, false, false);
#pragma unroll 1
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint64_t av = kdesc<64>(Vt, ks);
                mma_ss(tmem, av, mdesc<D>(Rt, ks), idK, ks > 0);
                mma_ss(tmem, av, mdesc<D>(Rt + 2 * D * D, ks), idK, 1);
                const uint64_t kh = kdesc<64>(Kt, ks), rh = kdesc<D>(Rt, ks);
                mma_ss(tmem + D, kh, rh, idV, ks > 0);
                mma_ss(tmem + D, kh, kdesc<D>(Rt + 2 * D * D, ks), idV, 1);
                if (kSplit) mma_ss(tmem + D, kdesc<64>(Kt + kC * D * 2, ks), rh, idV, 1);
            }
            mma_commit(bar_mma);
        }
        ok = __syncthreads_and(warp_wait(bar_mma, 0, a.err, kErrMma));
        tc_fence_after();
    }
    if (ok) {
        // warps 0-3: row j of d kt (+ its intra part + r) o phi'(k) -> dk;
        // warps 4-7: row j of d v (+ its intra part) -> dv.  16-byte accesses.
        const bool vside = warp >= 4;
        const int quarter = warp & 3, j = 16 * quarter + (lane & 15);
        const bool jv = lane < 16 && j < nvalid;
        const float* part = reinterpret_cast<const float*>(wsc + (vside ? L::kPV : L::kPK)) + j * D;
        const int64_t grow = (row0 + (int64_t)(jv ? j : 0) * a.Hkv) * D;
#pragma unroll 1
        for (int c32 = 0; c32 < D / 32; ++c32) {
            uint32_t x[32];
            tmem_ld32(tmem_addr(tmem + (vside ? D : 0), 32 * quarter, 32 * c32), x);
            tmem_ld_wait();
            reg_fence(x);
            if (jv) {
                float4 pp[8];
                uint4 kr[4];
#pragma unroll
                for (int q = 0; q < 8; ++q) pp[q] = reinterpret_cast<const float4*>(part + 32 * c32)[q];
                if (!vside) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) kr[q] = *reinterpret_cast<const uint4*>(a.k + grow + 32 * c32 + 8 * q);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float g[8], kx[8];
                    const float* pq = reinterpret_cast<const float*>(&pp[2 * q]);
                    if (!vside) unpack8(kr[q], kx);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        g[u] = __uint_as_float(x[8 * q + u]) + pq[u];
                        if (!vside) g[u] = (g[u] + rv[32 * c32 + 8 * q + u]) * dphi_fast(a.fmap, kx[u]);
                    }
                    const int64_t o = grow + 32 * c32 + 8 * q;
                    if (a.out_bf16)
                        store8(static_cast<__nv_bfloat16*>(vside ? a.dv : a.dk) + o, g);
                    else
                        store8(static_cast<float*>(vside ? a.dv : a.dk) + o, g);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 2 * D);
    }
}

template <int D, bool kSplit>
cudaError_t run(const BArgs& a, unsigned streams, cudaStream_t st) {
    static std::atomic<uint64_t> cfg_kv[kMaxDevices], cfg_mid[kMaxDevices], cfg_kg[kMaxDevices];
    cudaError_t e;
    if ((e = configure(bwd_kv_kernel<D, kSplit>, KvSmem<D, kSplit>::kBytes, cfg_kv)) != cudaSuccess) return e;
    if ((e = configure(bwd_mid_kernel<D, kSplit>, MidSmem<D>::kBytes, cfg_mid)) != cudaSuccess) return e;
    if ((e = configure(bwd_kvgrad_kernel<D, kSplit>, KgSmem<D>::kBytes, cfg_kg)) != cudaSuccess) return e;
    const unsigned chunks = streams * (unsigned)a.nc;
    const unsigned scan_grid = streams * (unsigned)scan_ctas<D>();
    bwd_kv_kernel<D, kSplit><<<chunks, 128, KvSmem<D, kSplit>::kBytes, st>>>(a);
    bwd_scan_kernel<D, false><<<scan_grid, kScanThreads, 0, st>>>(a);
    bwd_mid_kernel<D, kSplit><<<chunks, 256, MidSmem<D>::kBytes, st>>>(a);
    bwd_scan_kernel<D, true><<<scan_grid, kScanThreads, 0, st>>>(a);
    bwd_kvgrad_kernel<D, kSplit><<<chunks, 256, KgSmem<D>::kBytes, st>>>(a);
    note_launch(5);
    return cudaGetLastError();
}

static_assert(MidSmem<128>::kBytes <= 232448, "mid kernel shared memory");

}  // namespace bwd

bool backward_chunk_supported(const Problem& P) {
    if (P.gated || P.delta || P.decay_dim || P.mask || !P.io_bf16) return false;
    if (P.Dk != P.Dv || (P.Dk != 64 && P.Dk != 128)) return false;
    if (P.T < 1 || P.T > 0x7fffffffLL - 64) return false;
    const int64_t nc = (P.T + 63) / 64;
    const int64_t streams = P.B * P.Hkv;
    return streams * nc <= 0x7fffffffLL && streams * bwd::scan_ctas<128>() <= 0x7fffffffLL;
}

size_t backward_chunk_workspace_bytes(const Problem& P) {
    if (!backward_chunk_supported(P)) return 0;
    const size_t per = P.Dk == 64 ? bwd::Lay<64>::kChunk : bwd::Lay<128>::kChunk;
    return (size_t)P.B * P.Hkv * (size_t)((P.T + 63) / 64) * per;
}

cudaError_t backward_chunk_causal(const Problem& P, const void* q, const void* k, const void* v, const float* S0,
                                  const float* Z0, const void* dy, void* dq, void* dk, void* dv, float* dS0,
                                  float* dZ0, void* ws, cudaStream_t st) {
    using namespace bwd;
    unsigned* err = device_error_word();
    if (!err) return cudaErrorInvalidDevice;
    if (!q || !k || !v || !dy || !dq || !dk || !dv || !ws) return cudaErrorInvalidValue;
    BArgs a;
    memset(&a, 0, sizeof(a));
    a.B = (int)P.B;
    a.T = (int)P.T;
    a.Hq = P.Hq;
    a.Hkv = P.Hkv;
    a.G = P.G;
    a.nc = (int)((P.T + 63) / 64);
    a.fmap = P.fmap;
    a.norm = P.norm;
    a.out_bf16 = P.out_bf16;
    a.eps = P.eps;
    a.scale = P.scale;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.k = static_cast<const __nv_bfloat16*>(k);
    a.v = static_cast<const __nv_bfloat16*>(v);
    a.dy = static_cast<const __nv_bfloat16*>(dy);
    a.S0 = S0;
    a.Z0 = P.norm ? Z0 : nullptr;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.dS0 = dS0;
    a.dZ0 = P.norm ? dZ0 : nullptr;
    a.ws = static_cast<uint8_t*>(ws);
    a.err = err;
    const unsigned streams = (unsigned)(P.B * P.Hkv);
    // phi of elu + 1 and of relu + eps (x + eps is not a bf16 value in general)
    // enters as hi + lo; the identity of a bf16 input is exact in one part
    const bool split = P.fmap != LA_FMAP_NONE;
    if (P.Dk == 64) return split ? run<64, true>(a, streams, st) : run<64, false>(a, streams, st);
    return split ? run<128, true>(a, streams, st) : run<128, false>(a, streams, st);
}

}  // namespace la
