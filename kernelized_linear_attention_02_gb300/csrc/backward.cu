// backward.cu -- gradients of the causal pass (linear rule), on CUDA cores.
//
// "[Feature] LinearAttention layer for Keras", Mathematical definition /
// Causal: S_t = S_{t-1} + phi(k_t)^T v_t, Z_t = Z_{t-1} + phi(k_t),
// y_t = scale * phi(q_t) S_t / (phi(q_t) Z_t + eps) (without the normalizer
// the denominator is 1).  With a_t = phi(q_t), num_t = a_t S_t, den_t and the
// incoming gradient dy_t:
//   ds_t = scale dy_t / den_t                 gradient of num_t
//   dd_t = -(dy_t . y_t) / den_t              gradient of den_t (0 without the normalizer)
//   d a_t = S_t ds_t + dd_t Z_t               -> dq_t = d a_t * phi'(q_t)
// and, with R_t = sum_{i >= t} a_i ds_i^T (over the query heads of the kv
// head) and r_t = sum_{i >= t} a_i dd_i,
//   d phi(k_t) = R_t v_t + r_t                -> dk_t = d phi(k_t) * phi'(k_t)
//   dv_t = R_t^T phi(k_t)
//   dS0 = R_0, dZ0 = r_0.
// Pass 1 walks the tokens forward with (S, Z) and writes dq and (ds, dd) to
// the workspace; pass 2 walks them backward with (R, r) and writes dk, dv and
// the gradients of the initial state.  When few streams would leave most SMs
// idle, the sequence is cut into segments (blockIdx.y): an increment pass
// gives each segment's (dS, dZ) from zero, pass 1 folds the earlier
// segments' increments onto the initial state; a reverse increment pass gives
// each segment's (dR, dr), pass 2 starts from the sum over the later
// segments.  One CTA per (batch, kv head) stream and segment;
// warp w holds rows w, w + 8, ... of the Dk x Dv matrix, lane c columns c,
// c + 32, ... (Dk, Dv <= 128), as in the forward recurrence.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace la {

namespace {

constexpr int kThreads = 256;
constexpr int kRows = 16;  // rows per thread: Dk <= 128
constexpr int kCols = 4;   // columns per thread: Dv <= 128

struct BwdArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* S0;
    const float* Z0;
    const void* dy;
    void* dq;
    void* dk;
    void* dv;
    float* dS0;
    float* dZ0;
    float* ds;  // workspace (B, T, Hq, Dv)
    float* dd;  // workspace (B, T, Hq)
    Problem P;
    // sequence segments along blockIdx.y: steps [seg * cps, min(T, (seg + 1) * cps))
    int64_t cps;
    int nseg;
    float* S_seg;  // (B*Hkv, nseg, Dk, Dv) state increment of each segment
    float* Z_seg;  // (B*Hkv, nseg, Dk)
    float* R_seg;  // (B*Hkv, nseg, Dk, Dv) reverse increment sum_i a_i ds_i^T of each segment
    float* r_seg;  // (B*Hkv, nseg, Dk)
    int inc_only;  // increment pass: walk the segment from zero and write its increment only
};

// derivative of the feature map (Keras request, Feature maps): elu(x) + 1 has
// slope 1 for x > 0 and exp(x) below; relu(x) + eps has slope 1 for x > 0.
__device__ __forceinline__ float dphi(int fmap, float x) {
    if (fmap == LA_FMAP_ELU_PLUS_ONE) return x > 0.f ? 1.f : expf(x);
    if (fmap == LA_FMAP_RELU_EPS) return x > 0.f ? 1.f : 0.f;
    return 1.f;
}

// sum over the 32 lanes of a warp
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(kThreads) bwd_forward_kernel(BwdArgs a) {
    const Problem& P = a.P;
    const int Dk = P.Dk, Dv = P.Dv, G = P.G;
    __shared__ float fk[128], Zs[128], av[128], dsv[128], red[8][128];
    __shared__ float scal[2], red4[4];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t bh = blockIdx.x, b = bh / P.Hkv;
    const int hk = (int)(bh % P.Hkv);
    const TIn* q = static_cast<const TIn*>(a.q);
    const TIn* k = static_cast<const TIn*>(a.k);
    const TIn* v = static_cast<const TIn*>(a.v);
    const TIn* dy = static_cast<const TIn*>(a.dy);
    TOut* dq = static_cast<TOut*>(a.dq);

    const int seg = blockIdx.y;
    const int64_t t_begin = seg * a.cps, t_end = min(P.T, t_begin + a.cps);
    float s[kRows][kCols];
    const float* S0 = a.S0 && !a.inc_only ? a.S0 + bh * (int64_t)Dk * Dv : nullptr;
#pragma unroll
    for (int m = 0; m < kRows; ++m)
#pragma unroll
        for (int n = 0; n < kCols; ++n) {
            const int i = warp + 8 * m, j = lane + 32 * n;
            s[m][n] = (S0 && i < Dk && j < Dv) ? S0[(int64_t)i * Dv + j] : 0.f;
        }
    if (tid < 128) Zs[tid] = (P.norm && a.Z0 && !a.inc_only && tid < Dk) ? a.Z0[bh * Dk + tid] : 0.f;
    if (!a.inc_only)  // the state at the segment start: the earlier segments' increments
        for (int p = 0; p < seg; ++p) {
            const float* Sp = a.S_seg + ((int64_t)bh * a.nseg + p) * Dk * Dv;
#pragma unroll
            for (int m = 0; m < kRows; ++m)
#pragma unroll
                for (int n = 0; n < kCols; ++n) {
                    const int i = warp + 8 * m, j = lane + 32 * n;
                    if (i < Dk && j < Dv) s[m][n] += Sp[(int64_t)i * Dv + j];
                }
            if (P.norm && tid < Dk) Zs[tid] += a.Z_seg[((int64_t)bh * a.nseg + p) * Dk + tid];
        }
    __syncthreads();

    for (int64_t t = t_begin; t < t_end; ++t) {
        const int64_t tok = b * P.T + t;
        if (tid < Dk) fk[tid] = phi<false>(P.fmap, load_in(k, (tok * P.Hkv + hk) * Dk + tid), P.eps);
        float vj[kCols];
#pragma unroll
        for (int n = 0; n < kCols; ++n) {
            const int j = lane + 32 * n;
            vj[n] = j < Dv ? load_in(v, (tok * P.Hkv + hk) * Dv + j) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < kRows; ++m) {
            const int i = warp + 8 * m;
            const float f = i < Dk ? fk[i] : 0.f;
#pragma unroll
            for (int n = 0; n < kCols; ++n) s[m][n] = fmaf(f, vj[n], s[m][n]);
        }
        if (P.norm && tid < Dk) Zs[tid] += fk[tid];
        for (int r = 0; r < G && !a.inc_only; ++r) {
            const int64_t hq = tok * P.Hq + hk * G + r;
            __syncthreads();  // Zs and the previous head's av/dsv consumed
            if (tid < Dk) av[tid] = phi<false>(P.fmap, load_in(q, hq * Dk + tid), P.eps);
            __syncthreads();
            // num_j = sum_i a_i S_ij (across the warps' rows)
            float pn[kCols] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int m = 0; m < kRows; ++m) {
                const int i = warp + 8 * m;
                const float f = i < Dk ? av[i] : 0.f;
#pragma unroll
                for (int n = 0; n < kCols; ++n) pn[n] = fmaf(f, s[m][n], pn[n]);
            }
#pragma unroll
            for (int n = 0; n < kCols; ++n) red[warp][lane + 32 * n] = pn[n];
            if (warp == 0) {  // den = a . Z + eps
                float d = 0.f;
                for (int i = lane; i < Dk; i += 32) d = fmaf(av[i], Zs[i], d);
                d = warp_sum(d);
                if (lane == 0) scal[0] = P.norm ? d + P.eps : 1.f;
            }
            __syncthreads();
            const float den = scal[0];
            // ds_j = scale dy_j / den; dd = -(sum_j dy_j y_j) / den with y = scale num / den
            float part = 0.f;
            if (tid < Dv) {
                float num = 0.f;
#pragma unroll
                for (int w = 0; w < 8; ++w) num += red[w][tid];
                const float g = load_in(dy, hq * Dv + tid);
                const float dsj = P.scale * g / den;
                dsv[tid] = dsj;
                a.ds[hq * Dv + tid] = dsj;
                part = dsj * num;  // scale dy_j num_j / den
            }
            if (tid < 128) {  // warps 0..3
                part = warp_sum(part);
                if (lane == 0) red4[warp] = part;
            }
            __syncthreads();
            if (tid == 0) {
                const float sdn = red4[0] + red4[1] + red4[2] + red4[3];
                const float ddv = P.norm ? -sdn / den : 0.f;
                scal[1] = ddv;
                a.dd[hq] = ddv;
            }
            __syncthreads();
            const float ddv = scal[1];
            // d a_i = sum_j S_ij ds_j + dd Z_i (across the lanes' columns)
#pragma unroll
            for (int m = 0; m < kRows; ++m) {
                const int i = warp + 8 * m;
                float p = 0.f;
#pragma unroll
                for (int n = 0; n < kCols; ++n) {
                    const int j = lane + 32 * n;
                    p = fmaf(s[m][n], j < Dv ? dsv[j] : 0.f, p);
                }
                p = warp_sum(p);
                if (lane == 0 && i < Dk) {
                    const float da = p + ddv * Zs[i];
                    const float x = load_in(q, hq * Dk + i);
                    store_out(dq, hq * Dk + i, da * dphi(P.fmap, x));
                }
            }
        }
        __syncthreads();  // fk, av, dsv reused by the next token
    }
    if (a.inc_only) {  // this segment's state increment
        float* So = a.S_seg + ((int64_t)bh * a.nseg + seg) * Dk * Dv;
#pragma unroll
        for (int m = 0; m < kRows; ++m)
#pragma unroll
            for (int n = 0; n < kCols; ++n) {
                const int i = warp + 8 * m, j = lane + 32 * n;
                if (i < Dk && j < Dv) So[(int64_t)i * Dv + j] = s[m][n];
            }
        if (P.norm && tid < Dk) a.Z_seg[((int64_t)bh * a.nseg + seg) * Dk + tid] = Zs[tid];
    }
}

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(kThreads) bwd_reverse_kernel(BwdArgs a) {
    const Problem& P = a.P;
    const int Dk = P.Dk, Dv = P.Dv, G = P.G;
    __shared__ float fk[128], rs[128], red[8][128], av[8][128], dsv[8][128], ddv[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t bh = blockIdx.x, b = bh / P.Hkv;
    const int hk = (int)(bh % P.Hkv);
    const TIn* q = static_cast<const TIn*>(a.q);
    const TIn* k = static_cast<const TIn*>(a.k);
    const TIn* v = static_cast<const TIn*>(a.v);
    TOut* dk = static_cast<TOut*>(a.dk);
    TOut* dv = static_cast<TOut*>(a.dv);

    // segment `seg` of the reverse pass; the increment pass runs segments
    // 1 .. nseg-1 (blockIdx.y + 1), the full pass segments 0 .. nseg-1
    const int seg = blockIdx.y + (a.inc_only ? 1 : 0);
    const int64_t t_begin = seg * a.cps, t_end = min(P.T, t_begin + a.cps);
    float R[kRows][kCols];
#pragma unroll
    for (int m = 0; m < kRows; ++m)
#pragma unroll
        for (int n = 0; n < kCols; ++n) R[m][n] = 0.f;
    if (tid < 128) rs[tid] = 0.f;
    if (!a.inc_only)  // R at the segment end: the later segments' increments
        for (int p = seg + 1; p < a.nseg; ++p) {
            const float* Rp = a.R_seg + ((int64_t)bh * a.nseg + p) * Dk * Dv;
#pragma unroll
            for (int m = 0; m < kRows; ++m)
#pragma unroll
                for (int n = 0; n < kCols; ++n) {
                    const int i = warp + 8 * m, j = lane + 32 * n;
                    if (i < Dk && j < Dv) R[m][n] += Rp[(int64_t)i * Dv + j];
                }
            if (P.norm && tid < Dk) rs[tid] += a.r_seg[((int64_t)bh * a.nseg + p) * Dk + tid];
        }
    __syncthreads();

    for (int64_t t = t_end - 1; t >= t_begin; --t) {
        const int64_t tok = b * P.T + t;
        if (tid < Dk) fk[tid] = phi<false>(P.fmap, load_in(k, (tok * P.Hkv + hk) * Dk + tid), P.eps);
        float vj[kCols];
#pragma unroll
        for (int n = 0; n < kCols; ++n) {
            const int j = lane + 32 * n;
            vj[n] = j < Dv ? load_in(v, (tok * P.Hkv + hk) * Dv + j) : 0.f;
        }
        // R += sum over heads of a ds^T, r += sum a dd: heads in blocks of 8
        for (int r0 = 0; r0 < G; r0 += 8) {
            const int nh = min(8, G - r0);
            for (int idx = tid; idx < nh * 128; idx += kThreads) {
                const int rr = idx >> 7, e = idx & 127;
                const int64_t hq = tok * P.Hq + hk * G + r0 + rr;
                av[rr][e] = e < Dk ? phi<false>(P.fmap, load_in(q, hq * Dk + e), P.eps) : 0.f;
                dsv[rr][e] = e < Dv ? a.ds[hq * Dv + e] : 0.f;
            }
            if (tid < nh) ddv[tid] = a.dd[tok * P.Hq + hk * G + r0 + tid];
            __syncthreads();
            for (int rr = 0; rr < nh; ++rr) {
#pragma unroll
                for (int m = 0; m < kRows; ++m) {
                    const float f = av[rr][warp + 8 * m];
#pragma unroll
                    for (int n = 0; n < kCols; ++n) R[m][n] = fmaf(f, dsv[rr][lane + 32 * n], R[m][n]);
                }
                if (P.norm && tid < Dk) rs[tid] = fmaf(av[rr][tid], ddv[rr], rs[tid]);
            }
            __syncthreads();  // av / dsv reused by the next block of heads
        }
        if (a.inc_only) continue;  // uniform: the increment pass needs no outputs
        // d phi(k)_i = sum_j R_ij v_j + r_i (across lanes); dv_j = sum_i R_ij phi(k)_i (across warps)
        float pv[kCols] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < kRows; ++m) {
            const int i = warp + 8 * m;
            const float f = i < Dk ? fk[i] : 0.f;
            float p = 0.f;
#pragma unroll
            for (int n = 0; n < kCols; ++n) {
                p = fmaf(R[m][n], vj[n], p);
                pv[n] = fmaf(R[m][n], f, pv[n]);
            }
            p = warp_sum(p);
            if (lane == 0 && i < Dk) {
                const float dfk = p + (P.norm ? rs[i] : 0.f);
                const float x = load_in(k, (tok * P.Hkv + hk) * Dk + i);
                store_out(dk, (tok * P.Hkv + hk) * Dk + i, dfk * dphi(P.fmap, x));
            }
        }
#pragma unroll
        for (int n = 0; n < kCols; ++n) red[warp][lane + 32 * n] = pv[n];
        __syncthreads();
        if (tid < Dv) {
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) acc += red[w][tid];
            store_out(dv, (tok * P.Hkv + hk) * Dv + tid, acc);
        }
        __syncthreads();  // fk, red, rs reused by the previous token
    }
    if (a.inc_only) {  // this segment's reverse increment
        float* o = a.R_seg + ((int64_t)bh * a.nseg + seg) * Dk * Dv;
#pragma unroll
        for (int m = 0; m < kRows; ++m)
#pragma unroll
            for (int n = 0; n < kCols; ++n) {
                const int i = warp + 8 * m, j = lane + 32 * n;
                if (i < Dk && j < Dv) o[(int64_t)i * Dv + j] = R[m][n];
            }
        if (P.norm && tid < Dk) a.r_seg[((int64_t)bh * a.nseg + seg) * Dk + tid] = rs[tid];
        return;
    }
    if (a.dS0 && seg == 0) {
        float* o = a.dS0 + bh * (int64_t)Dk * Dv;
#pragma unroll
        for (int m = 0; m < kRows; ++m)
#pragma unroll
            for (int n = 0; n < kCols; ++n) {
                const int i = warp + 8 * m, j = lane + 32 * n;
                if (i < Dk && j < Dv) o[(int64_t)i * Dv + j] = R[m][n];
            }
    }
    if (a.dZ0 && P.norm && seg == 0 && tid < Dk) a.dZ0[bh * Dk + tid] = rs[tid];
}

template <typename TIn, typename TOut>
cudaError_t launch(const BwdArgs& a, cudaStream_t st) {
    const unsigned streams = (unsigned)(a.P.B * a.P.Hkv);
    auto run = [&](auto kern, const BwdArgs& x, int ny) -> cudaError_t {
        kern<<<dim3(streams, (unsigned)ny), kThreads, 0, st>>>(x);
        note_launch();
        return cudaGetLastError();
    };
    cudaError_t e;
    if (a.nseg > 1) {  // increments of segments 0 .. nseg-2 (forward)
        BwdArgs x = a;
        x.inc_only = 1;
        if ((e = run(bwd_forward_kernel<TIn, TOut>, x, a.nseg - 1)) != cudaSuccess) return e;
    }
    if ((e = run(bwd_forward_kernel<TIn, TOut>, a, a.nseg)) != cudaSuccess) return e;
    if (a.nseg > 1) {  // reverse increments of segments 1 .. nseg-1
        BwdArgs x = a;
        x.inc_only = 1;
        if ((e = run(bwd_reverse_kernel<TIn, TOut>, x, a.nseg - 1)) != cudaSuccess) return e;
    }
    return run(bwd_reverse_kernel<TIn, TOut>, a, a.nseg);
}

// Segments: enough to give most SMs a CTA when the streams alone do not, at
// least 256 steps each, at most 8 MiB of segment scratch.
constexpr size_t kSegCap = (size_t)8 << 20;
size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

int bwd_segments(const Problem& P) {
    if (P.T < 512) return 1;
    const int64_t streams = P.B * P.Hkv;
    const int sms = device_sm_count();
    if (sms <= 0 || streams * 2 > sms) return 1;
    int64_t n = std::min<int64_t>(sms / streams, P.T / 256);
    const size_t per = sizeof(float) * (size_t)streams * (2 * (size_t)P.Dk * P.Dv + 2 * (size_t)P.Dk);
    n = std::min<int64_t>(n, (int64_t)(kSegCap / per));
    if (n < 2) return 1;
    const int64_t cps = (P.T + n - 1) / n;
    return (int)((P.T + cps - 1) / cps);
}

struct BwdLayout {
    size_t ds, dd, S, Z, R, r, total;
};
BwdLayout bwd_layout(const Problem& P, int nseg) {
    const size_t n = (size_t)P.B * P.T * P.Hq, streams = (size_t)(P.B * P.Hkv);
    BwdLayout L{};
    L.ds = 0;
    L.dd = up256(sizeof(float) * n * P.Dv);
    L.S = L.dd + up256(sizeof(float) * n);
    if (nseg <= 1) {
        L.Z = L.R = L.r = L.total = L.S;
        return L;
    }
    L.Z = L.S + up256(sizeof(float) * streams * nseg * P.Dk * P.Dv);
    L.R = L.Z + up256(sizeof(float) * streams * nseg * P.Dk);
    L.r = L.R + up256(sizeof(float) * streams * nseg * P.Dk * P.Dv);
    L.total = L.r + up256(sizeof(float) * streams * nseg * P.Dk);
    return L;
}

}  // namespace

size_t backward_workspace_bytes(const Problem& P) {
    // covers both paths: the chunk form runs unless the pointers are not 16-byte aligned
    return std::max(bwd_layout(P, bwd_segments(P)).total, backward_chunk_workspace_bytes(P));
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

cudaError_t backward_causal(const Problem& P, const void* q, const void* k, const void* v, const float* S0,
                            const float* Z0, const void* dy, void* dq, void* dk, void* dv, float* dS0, float* dZ0,
                            void* ws, cudaStream_t st) {
    if (backward_chunk_supported(P) && aligned16(q) && aligned16(k) && aligned16(v) && aligned16(dy) &&
        aligned16(dq) && aligned16(dk) && aligned16(dv) && aligned16(ws))
        return backward_chunk_causal(P, q, k, v, S0, Z0, dy, dq, dk, dv, dS0, dZ0, ws, st);
    BwdArgs a{};
    a.q = q, a.k = k, a.v = v, a.S0 = S0, a.Z0 = P.norm ? Z0 : nullptr, a.dy = dy;
    a.dq = dq, a.dk = dk, a.dv = dv, a.dS0 = dS0, a.dZ0 = P.norm ? dZ0 : nullptr;
    a.P = P;
    a.nseg = bwd_segments(P);
    a.cps = (P.T + a.nseg - 1) / a.nseg;
    const BwdLayout L = bwd_layout(P, a.nseg);
    char* w = static_cast<char*>(ws);
    a.ds = reinterpret_cast<float*>(w + L.ds);
    a.dd = reinterpret_cast<float*>(w + L.dd);
    if (a.nseg > 1) {
        a.S_seg = reinterpret_cast<float*>(w + L.S);
        a.Z_seg = reinterpret_cast<float*>(w + L.Z);
        a.R_seg = reinterpret_cast<float*>(w + L.R);
        a.r_seg = reinterpret_cast<float*>(w + L.r);
    }
    if (P.io_bf16)
        return P.out_bf16 ? launch<__nv_bfloat16, __nv_bfloat16>(a, st) : launch<__nv_bfloat16, float>(a, st);
    return P.out_bf16 ? launch<float, __nv_bfloat16>(a, st) : launch<float, float>(a, st);
}

}  // namespace la
