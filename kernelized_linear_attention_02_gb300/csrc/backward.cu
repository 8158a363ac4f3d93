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
// the gradients of the initial state.  One CTA per (batch, kv head) stream;
// warp w holds rows w, w + 8, ... of the Dk x Dv matrix, lane c columns c,
// c + 32, ... (Dk, Dv <= 128), as in the forward recurrence.
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

    float s[kRows][kCols];
    const float* S0 = a.S0 ? a.S0 + bh * (int64_t)Dk * Dv : nullptr;
#pragma unroll
    for (int m = 0; m < kRows; ++m)
#pragma unroll
        for (int n = 0; n < kCols; ++n) {
            const int i = warp + 8 * m, j = lane + 32 * n;
            s[m][n] = (S0 && i < Dk && j < Dv) ? S0[(int64_t)i * Dv + j] : 0.f;
        }
    if (tid < 128) Zs[tid] = (P.norm && a.Z0 && tid < Dk) ? a.Z0[bh * Dk + tid] : 0.f;
    __syncthreads();

    for (int64_t t = 0; t < P.T; ++t) {
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
        for (int r = 0; r < G; ++r) {
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

    float R[kRows][kCols];
#pragma unroll
    for (int m = 0; m < kRows; ++m)
#pragma unroll
        for (int n = 0; n < kCols; ++n) R[m][n] = 0.f;
    if (tid < 128) rs[tid] = 0.f;
    __syncthreads();

    for (int64_t t = P.T - 1; t >= 0; --t) {
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
    if (a.dS0) {
        float* o = a.dS0 + bh * (int64_t)Dk * Dv;
#pragma unroll
        for (int m = 0; m < kRows; ++m)
#pragma unroll
            for (int n = 0; n < kCols; ++n) {
                const int i = warp + 8 * m, j = lane + 32 * n;
                if (i < Dk && j < Dv) o[(int64_t)i * Dv + j] = R[m][n];
            }
    }
    if (a.dZ0 && P.norm && tid < Dk) a.dZ0[bh * Dk + tid] = rs[tid];
}

template <typename TIn, typename TOut>
cudaError_t launch(const BwdArgs& a, cudaStream_t st) {
    const dim3 grid((unsigned)(a.P.B * a.P.Hkv));
    bwd_forward_kernel<TIn, TOut><<<grid, kThreads, 0, st>>>(a);
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_reverse_kernel<TIn, TOut><<<grid, kThreads, 0, st>>>(a);
    note_launch();
    return cudaGetLastError();
}

}  // namespace

size_t backward_workspace_bytes(const Problem& P) {
    const size_t n = (size_t)P.B * P.T * P.Hq;
    return ((sizeof(float) * n * P.Dv + 255) & ~(size_t)255) + sizeof(float) * n;
}

cudaError_t backward_causal(const Problem& P, const void* q, const void* k, const void* v, const float* S0,
                            const float* Z0, const void* dy, void* dq, void* dk, void* dv, float* dS0, float* dZ0,
                            void* ws, cudaStream_t st) {
    BwdArgs a{};
    a.q = q, a.k = k, a.v = v, a.S0 = S0, a.Z0 = P.norm ? Z0 : nullptr, a.dy = dy;
    a.dq = dq, a.dk = dk, a.dv = dv, a.dS0 = dS0, a.dZ0 = P.norm ? dZ0 : nullptr;
    const size_t n = (size_t)P.B * P.T * P.Hq;
    a.ds = static_cast<float*>(ws);
    a.dd = reinterpret_cast<float*>(static_cast<char*>(ws) + ((sizeof(float) * n * P.Dv + 255) & ~(size_t)255));
    a.P = P;
    if (P.io_bf16)
        return P.out_bf16 ? launch<__nv_bfloat16, __nv_bfloat16>(a, st) : launch<__nv_bfloat16, float>(a, st);
    return P.out_bf16 ? launch<float, __nv_bfloat16>(a, st) : launch<float, float>(a, st);
}

}  // namespace la
