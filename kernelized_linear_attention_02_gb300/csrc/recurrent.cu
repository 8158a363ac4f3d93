// recurrent.cu -- the token-by-token recurrence on CUDA cores.
//
// This is the float32 path of the library (float32 q/k/v need float32
// products, which the bf16 tensor-core kernels do not give) and the path for
// shapes the tensor-core kernels do not cover.  One CTA owns one (batch,
// kv-head) state stream and walks its tokens in order, exactly the causal
// recurrence of the Keras request ("Mathematical definition / Causal"):
// update S and Z with token t first, then read out every query head of the
// group with S_t ("the current token is included in its own context").
//
// The same kernel also runs the two halves of the non-causal form: a state
// pass (update only; S = sum_j phi(K_j)^T V_j, Z = sum_j phi(K_j)) and a
// read-out pass with that fixed global state.
//
// Few (batch, kv-head) streams would leave most SMs idle, so a long sequence
// is cut into segments (blockIdx.y), as the chunk kernel does: a state pass
// gives each segment's state and key-sum increment from a zero state and its
// summed log decay per key dimension; the causal pass then folds the earlier
// segments onto the initial state in order (S <- exp(G_seg) S + dS_seg, Z <-
// Z + dZ_seg), which is the recurrence regrouped, and walks its own steps.
//
// The delta rules of the ONNX-light operator decay the state first, then add
// beta k (x) (v - S^T k): the residual needs S^T k of the decayed state, a
// reduction over the key dimensions held by the eight warps (one exchange
// through shared memory per step).  Their update is not additive in S, so
// they never take the segment split.
//
// A sequence-validity mask (Keras request, Masking) skips the update of an
// invalid step (the state passes through unchanged, no decay either) and
// writes zeros for its outputs.  The mask is per (batch, step), so the
// decision is uniform across the CTA.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace la {

namespace {

constexpr int kThreads = 256;  // 8 warps: warp w owns rows w, w+8, ...; lane c owns columns c, c+32, ...
constexpr int kRowsPerThread = 16;  // Dk <= 128
constexpr int kColsPerThread = 4;   // Dv <= 128
constexpr int kHeadBlock = 4;       // query heads reduced per round

struct RecArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* decay;
    const float* S0;
    const float* Z0;
    void* y;
    float* S_out;
    float* Z_out;
    Problem P;
    int mode;  // kModeCausal, kModeStateOnly, kModeReadoutOnly
    // sequence segments along blockIdx.y: steps [seg * cps, min(T, (seg + 1) * cps))
    int64_t cps = 0;         // 0: one segment of all T steps
    int nseg = 1;
    float* S_seg = nullptr;  // (B*Hkv, nseg, Dk, Dv) state increment of each segment
    float* Z_seg = nullptr;  // (B*Hkv, nseg, Dk) key-sum increment
    float* G_seg = nullptr;  // (B*Hkv, nseg, Dk) summed log decay per key dimension (gated)
    const void* beta = nullptr;  // delta rules: (B, T, Hkv) or (B, T, 1)
    int beta_per_head = 1;
};

enum { kModeCausal = 0, kModeStateOnly = 1, kModeReadoutOnly = 2 };

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(kThreads) recurrent_kernel(RecArgs a) {
    const Problem& P = a.P;
    const int Dk = P.Dk, Dv = P.Dv, G = P.G;
    extern __shared__ float smem[];
    float* fk = smem;             // [128]   phi(k_t)
    float* Zs = fk + 128;         // [128]   Z_t
    float* den = Zs + 128;        // [128]   phi(q).Z + eps per query head of the group
    float* fq = den + 128;        // [G*Dk]  phi(q_t) of the group
    float* red = fq + G * Dk;     // [kHeadBlock][8][128] partial read-outs

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t bh = blockIdx.x;
    const int64_t b = bh / P.Hkv;
    const int hk = (int)(bh % P.Hkv);
    const TIn* q = static_cast<const TIn*>(a.q);
    const TIn* k = static_cast<const TIn*>(a.k);
    const TIn* v = static_cast<const TIn*>(a.v);
    const TIn* decay = static_cast<const TIn*>(a.decay);
    const TIn* beta = static_cast<const TIn*>(a.beta);
    TOut* y = static_cast<TOut*>(a.y);
    const bool update = a.mode != kModeReadoutOnly;
    const bool readout = a.mode != kModeStateOnly;
    const int seg = blockIdx.y;
    const int64_t t_begin = a.cps ? seg * a.cps : 0;
    const int64_t t_end = a.cps ? min(P.T, t_begin + a.cps) : P.T;
    const bool seg_state = a.mode == kModeStateOnly && a.S_seg;          // this segment's increment
    const bool seg_fold = a.mode == kModeCausal && a.S_seg && seg > 0;  // earlier segments folded in
    const bool last_seg = seg == a.nseg - 1;

    // state slice owned by this thread: rows warp + 8m, columns lane + 32n
    float s[kRowsPerThread][kColsPerThread];
    float gl[kRowsPerThread];  // segment state pass: summed log decay of rows warp + 8m
    const float* S0 = a.S0 && !seg_state ? a.S0 + bh * (int64_t)Dk * Dv : nullptr;
#pragma unroll
    for (int m = 0; m < kRowsPerThread; ++m) {
        gl[m] = 0.f;
#pragma unroll
        for (int n = 0; n < kColsPerThread; ++n) {
            const int i = warp + 8 * m, j = lane + 32 * n;
            s[m][n] = (S0 && i < Dk && j < Dv) ? S0[(int64_t)i * Dv + j] : 0.f;
        }
    }
    if (tid < 128) Zs[tid] = (P.norm && a.Z0 && !seg_state && tid < Dk) ? a.Z0[bh * Dk + tid] : 0.f;
    if (seg_fold) {
        // start state of this segment: the earlier segments in order
        for (int p = 0; p < seg; ++p) {
            const float* Sp = a.S_seg + ((int64_t)bh * a.nseg + p) * Dk * Dv;
            const float* Gp = a.G_seg + ((int64_t)bh * a.nseg + p) * Dk;
#pragma unroll
            for (int m = 0; m < kRowsPerThread; ++m) {
                const int i = warp + 8 * m;
                if (i >= Dk) continue;
                const float e = P.gated ? expf(Gp[i]) : 1.f;
#pragma unroll
                for (int n = 0; n < kColsPerThread; ++n) {
                    const int j = lane + 32 * n;
                    if (j < Dv) s[m][n] = fmaf(e, s[m][n], Sp[(int64_t)i * Dv + j]);
                }
            }
            if (P.norm && tid < Dk) Zs[tid] += a.Z_seg[((int64_t)bh * a.nseg + p) * Dk + tid];
        }
    }
    __syncthreads();  // Z0 may alias Z_out of this same CTA only

    for (int64_t t = t_begin; t < t_end; ++t) {
        const int64_t tok = b * P.T + t;
        if (!step_valid(P.mask, tok)) {
            if (readout)
                for (int idx = tid; idx < G * Dv; idx += kThreads)
                    store_out(y, (tok * P.Hq + hk * G) * Dv + idx, 0.f);
            continue;
        }
        if (update)
            for (int i = tid; i < Dk; i += kThreads)
                fk[i] = phi<false>(P.fmap, load_in(k, (tok * P.Hkv + hk) * Dk + i), P.eps);
        if (readout)
            for (int idx = tid; idx < G * Dk; idx += kThreads) {
                const int r = idx / Dk, i = idx - r * Dk;
                fq[idx] = phi<false>(P.fmap, load_in(q, (tok * P.Hq + hk * G + r) * Dk + i), P.eps);
            }
        __syncthreads();

        if (update) {
            // decay of this step: one per kv head, or one per key dimension (row of S)
            const float gh = P.gated && !P.decay_dim ? load_in(decay, tok * P.Hkv + hk) : 0.f;
            const float dec = P.gated && !P.decay_dim ? expf(gh) : 1.f;
            float vj[kColsPerThread];
#pragma unroll
            for (int n = 0; n < kColsPerThread; ++n) {
                const int j = lane + 32 * n;
                vj[n] = j < Dv ? load_in(v, (tok * P.Hkv + hk) * Dv + j) : 0.f;
            }
            if (P.delta) {
                // decay, then u = beta (v - S^T k) with the decayed S, then S += k (x) u
                float pn[kColsPerThread] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int m = 0; m < kRowsPerThread; ++m) {
                    const int i = warp + 8 * m;
                    const float f = i < Dk ? fk[i] : 0.f;
                    const float gi = P.gated && P.decay_dim && i < Dk ? load_in(decay, (tok * P.Hkv + hk) * Dk + i) : gh;
                    const float di = P.gated && P.decay_dim ? expf(gi) : dec;
#pragma unroll
                    for (int n = 0; n < kColsPerThread; ++n) {
                        s[m][n] *= di;
                        pn[n] = fmaf(s[m][n], f, pn[n]);
                    }
                }
#pragma unroll
                for (int n = 0; n < kColsPerThread; ++n) red[warp * 128 + lane + 32 * n] = pn[n];
                __syncthreads();
                const float bt = load_in(beta, a.beta_per_head ? tok * P.Hkv + hk : tok);
                float un[kColsPerThread];
#pragma unroll
                for (int n = 0; n < kColsPerThread; ++n) {
                    const int j = lane + 32 * n;
                    float acc = 0.f;
#pragma unroll
                    for (int w = 0; w < 8; ++w) acc += red[w * 128 + j];
                    un[n] = bt * (vj[n] - acc);
                }
#pragma unroll
                for (int m = 0; m < kRowsPerThread; ++m) {
                    const int i = warp + 8 * m;
                    const float f = i < Dk ? fk[i] : 0.f;
#pragma unroll
                    for (int n = 0; n < kColsPerThread; ++n) s[m][n] = fmaf(f, un[n], s[m][n]);
                }
            } else {
#pragma unroll
                for (int m = 0; m < kRowsPerThread; ++m) {
                    const int i = warp + 8 * m;
                    const float f = i < Dk ? fk[i] : 0.f;
                    const float gi = P.gated && P.decay_dim && i < Dk ? load_in(decay, (tok * P.Hkv + hk) * Dk + i) : gh;
                    const float di = P.gated && P.decay_dim ? expf(gi) : dec;
                    gl[m] += gi;
#pragma unroll
                    for (int n = 0; n < kColsPerThread; ++n) s[m][n] = fmaf(f, vj[n], di * s[m][n]);
                }
            }
            if (P.norm && tid < Dk) Zs[tid] += fk[tid];
        }
        __syncthreads();          // Zs complete; fk consumed before the next token overwrites it
        if (!readout) continue;  // uniform across the CTA

        if (P.norm)
            for (int r = warp; r < G; r += 8) {
                float d = 0.f;
                for (int i = lane; i < Dk; i += 32) d = fmaf(fq[r * Dk + i], Zs[i], d);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
                if (lane == 0) den[r] = d + P.eps;
            }
        for (int r0 = 0; r0 < G; r0 += kHeadBlock) {
            const int nh = min(kHeadBlock, G - r0);
            for (int rr = 0; rr < nh; ++rr) {
                float acc[kColsPerThread] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int m = 0; m < kRowsPerThread; ++m) {
                    const int i = warp + 8 * m;
                    const float f = i < Dk ? fq[(r0 + rr) * Dk + i] : 0.f;
#pragma unroll
                    for (int n = 0; n < kColsPerThread; ++n) acc[n] = fmaf(f, s[m][n], acc[n]);
                }
#pragma unroll
                for (int n = 0; n < kColsPerThread; ++n)
                    red[(rr * 8 + warp) * 128 + lane + 32 * n] = acc[n];
            }
            __syncthreads();  // red and den complete
            for (int idx = tid; idx < nh * Dv; idx += kThreads) {
                const int rr = idx / Dv, j = idx - rr * Dv;
                float num = 0.f;
#pragma unroll
                for (int w = 0; w < 8; ++w) num += red[(rr * 8 + w) * 128 + j];
                const float out = P.norm ? num / den[r0 + rr] : num;
                store_out(y, (tok * P.Hq + hk * G + r0 + rr) * Dv + j, P.scale * out);
            }
            __syncthreads();  // red is reused by the next head block / token
        }
    }

    // the segment's increment (state pass), or the final state (last segment)
    float* So = seg_state ? a.S_seg + ((int64_t)bh * a.nseg + seg) * Dk * Dv
                          : (a.S_out && last_seg ? a.S_out + bh * (int64_t)Dk * Dv : nullptr);
    float* Zo = seg_state ? (a.Z_seg ? a.Z_seg + ((int64_t)bh * a.nseg + seg) * Dk : nullptr)
                          : (a.Z_out && last_seg ? a.Z_out + bh * Dk : nullptr);
    if (So) {
#pragma unroll
        for (int m = 0; m < kRowsPerThread; ++m)
#pragma unroll
            for (int n = 0; n < kColsPerThread; ++n) {
                const int i = warp + 8 * m, j = lane + 32 * n;
                if (i < Dk && j < Dv) So[(int64_t)i * Dv + j] = s[m][n];
            }
    }
    if (seg_state && a.G_seg && lane == 0)
#pragma unroll
        for (int m = 0; m < kRowsPerThread; ++m) {
            const int i = warp + 8 * m;
            if (i < Dk) a.G_seg[((int64_t)bh * a.nseg + seg) * Dk + i] = gl[m];
        }
    __syncthreads();
    if (Zo && P.norm && tid < Dk) Zo[tid] = Zs[tid];
}

template <typename TIn, typename TOut>
cudaError_t launch(const RecArgs& a, int ny, cudaStream_t st) {
    const Problem& P = a.P;
    const size_t smem = sizeof(float) * (3 * 128 + (size_t)P.G * P.Dk + kHeadBlock * 8 * 128);
    auto kern = recurrent_kernel<TIn, TOut>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)(P.B * P.Hkv), (unsigned)ny), kThreads, smem, st>>>(a);
    note_launch();
    return cudaGetLastError();
}

cudaError_t dispatch(const RecArgs& a, cudaStream_t st, int ny = 1) {
    if (a.P.io_bf16)
        return a.P.out_bf16 ? launch<__nv_bfloat16, __nv_bfloat16>(a, ny, st)
                            : launch<__nv_bfloat16, float>(a, ny, st);
    return a.P.out_bf16 ? launch<float, __nv_bfloat16>(a, ny, st) : launch<float, float>(a, ny, st);
}

// Segments of the recurrence: enough to give most SMs a CTA when the
// streams alone do not, at least 256 steps each, and scratch of at most
// 8 MiB.
constexpr size_t kSegScratchCap = (size_t)8 << 20;
constexpr size_t kWsAlign = 256;
size_t up256(size_t x) { return (x + kWsAlign - 1) & ~(kWsAlign - 1); }

int rec_segments(const Problem& P) {
    if (P.T < 512 || P.delta) return 1;
    const int64_t streams = P.B * P.Hkv;
    const int sms = device_sm_count();
    if (sms <= 0 || streams * 2 > sms) return 1;
    int64_t n = std::min<int64_t>(sms / streams, P.T / 256);
    const size_t per = sizeof(float) * (size_t)streams * ((size_t)P.Dk * P.Dv + 2 * (size_t)P.Dk);
    n = std::min<int64_t>(n, (int64_t)(kSegScratchCap / per));
    if (n < 2) return 1;
    const int64_t cps = (P.T + n - 1) / n;
    return (int)((P.T + cps - 1) / cps);  // no empty segment
}

struct SegLayout {
    size_t S, Z, G, S0, Z0, total;
};
SegLayout seg_layout(const Problem& P, int nseg) {
    const size_t streams = (size_t)(P.B * P.Hkv);
    SegLayout L{};
    L.S = 0;
    L.Z = L.S + up256(sizeof(float) * streams * nseg * P.Dk * P.Dv);
    L.G = L.Z + up256(sizeof(float) * streams * nseg * P.Dk);
    L.S0 = L.G + up256(sizeof(float) * streams * nseg * P.Dk);
    L.Z0 = L.S0 + up256(sizeof(float) * streams * P.Dk * P.Dv);
    L.total = L.Z0 + up256(sizeof(float) * streams * P.Dk);
    return L;
}

}  // namespace

size_t recurrent_smem_bytes(const Problem& P) {
    return sizeof(float) * (3 * 128 + (size_t)P.G * P.Dk + kHeadBlock * 8 * 128);
}

size_t recurrent_workspace_bytes(const Problem& P) {
    const int nseg = rec_segments(P);
    return nseg > 1 ? seg_layout(P, nseg).total : 0;
}

cudaError_t recurrent_causal(const Problem& P, const void* q, const void* k, const void* v,
                             const void* decay, const float* S0, const float* Z0, void* y,
                             float* S_out, float* Z_out, cudaStream_t st, void* ws, size_t ws_bytes) {
    RecArgs a{q, k, v, decay, S0, Z0, y, S_out, Z_out, P, kModeCausal};
    const int nseg = rec_segments(P);
    if (nseg <= 1 || !ws || ws_bytes < seg_layout(P, nseg).total) return dispatch(a, st);
    const SegLayout L = seg_layout(P, nseg);
    char* w = static_cast<char*>(ws);
    const size_t streams = (size_t)(P.B * P.Hkv);
    // a final state written over the initial one: the segments read a copy
    if (S0 && S0 == S_out) {
        cudaError_t e = cudaMemcpyAsync(w + L.S0, S0, sizeof(float) * streams * P.Dk * P.Dv,
                                        cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess) return e;
        a.S0 = reinterpret_cast<const float*>(w + L.S0);
    }
    if (Z0 && Z0 == Z_out) {
        cudaError_t e = cudaMemcpyAsync(w + L.Z0, Z0, sizeof(float) * streams * P.Dk, cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess) return e;
        a.Z0 = reinterpret_cast<const float*>(w + L.Z0);
    }
    a.cps = (P.T + nseg - 1) / nseg;
    a.nseg = nseg;
    a.S_seg = reinterpret_cast<float*>(w + L.S);
    a.Z_seg = P.norm ? reinterpret_cast<float*>(w + L.Z) : nullptr;
    a.G_seg = reinterpret_cast<float*>(w + L.G);
    // pass 1: increments of segments 0 .. nseg-2; pass 2: every segment's outputs
    RecArgs a1 = a;
    a1.q = nullptr;
    a1.y = nullptr;
    a1.S0 = a1.Z0 = nullptr;
    a1.S_out = a1.Z_out = nullptr;
    a1.mode = kModeStateOnly;
    cudaError_t e = dispatch(a1, st, nseg - 1);
    if (e != cudaSuccess) return e;
    return dispatch(a, st, nseg);
}

cudaError_t recurrent_delta(const Problem& P, const void* q, const void* k, const void* v, const void* decay,
                            const void* beta, int beta_per_head, const float* S0, void* y, float* S_out,
                            cudaStream_t st) {
    RecArgs a{q, k, v, decay, S0, nullptr, y, S_out, nullptr, P, kModeCausal};
    a.P.norm = 0;
    a.beta = beta;
    a.beta_per_head = beta_per_head;
    return dispatch(a, st);
}

cudaError_t recurrent_noncausal(const Problem& P, const void* q, const void* k, const void* v,
                                void* y, float* S_ws, float* Z_ws, cudaStream_t st) {
    // pass 1: global state; pass 2: read-out with it (no update)
    RecArgs a1{nullptr, k, v, nullptr, nullptr, nullptr, nullptr, S_ws, Z_ws, P, kModeStateOnly};
    a1.P.gated = 0;
    cudaError_t e = dispatch(a1, st);
    if (e != cudaSuccess) return e;
    RecArgs a2{q, nullptr, nullptr, nullptr, S_ws, Z_ws, y, nullptr, nullptr, P, kModeReadoutOnly};
    a2.P.gated = 0;
    return dispatch(a2, st);
}

}  // namespace la
