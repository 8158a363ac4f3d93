// chunk_host.cu -- host orchestration of the tensor-core path: sequence
// segmentation, workspace layout, tensor maps, and the small CUDA-core
// kernel that sums the per-segment states of the non-causal form.
//
// Causal, sequence split into P segments per (batch, kv head):
//   pass 1 (state mode, segments 0..P-2): dS_p, dZ_p, log decay of segment p
//   pass 2 (causal mode, all segments): each CTA folds dS_0..dS_{s-1} onto
//          the initial state (decay-weighted) to get the start state of its
//          segment, then produces its outputs; the last segment writes the
//          final state
// Non-causal: pass 1 over all segments, sum, then the read-out pass.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <utility>

#include "chunk_args.h"
#include "kernels.h"
#include "tma_host.h"

namespace la {

__device__ unsigned int g_chunk_err = 0;

namespace {

constexpr size_t kAlign = 256;
size_t round_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

struct DevInfo {
    int sms = 0;
    unsigned* err = nullptr;
    uint64_t ctx = 0;  // context the entry was filled in
};

// SM count and error-word address of the current device, looked up once per
// device and context (a device reset gives the device a new context, whose
// symbol addresses are looked up again).
bool dev_info(DevInfo* out) {
    static std::mutex mu;
    static DevInfo info[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    const uint64_t ctx = current_context_id();
    std::lock_guard<std::mutex> lk(mu);
    if (!info[dev].err || ctx == 0 || info[dev].ctx != ctx) {
        int sms = 0;
        void* p = nullptr;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
        // also makes the device's primary context current if none was
        if (cudaGetSymbolAddress(&p, g_chunk_err) != cudaSuccess) return false;
        info[dev].sms = sms;
        info[dev].err = static_cast<unsigned*>(p);
        info[dev].ctx = current_context_id();
    }
    *out = info[dev];
    return true;
}

struct Plan {
    int nseg, cps;
    int sub = 1;  // causal: state-pass sub-segments per segment
};

// Enough (batch, kv head, segment) tiles for one CTA per SM, never more
// segments than chunks.
Plan plan_segments(int64_t BH, int nchunks, int sms) {
    int nseg = BH >= sms ? 1 : std::max<int>(1, static_cast<int>(sms / BH));
    nseg = std::min(nseg, nchunks);
    const int cps = (nchunks + nseg - 1) / nseg;
    return {(nchunks + cps - 1) / cps, cps};
}

// Causal plan.  At head size 64 the linear rule's state pass runs two CTAs
// per SM (chunk.cuh, Cfg::kTwoPerSm), so it takes each full segment as two
// half-length sub-segments whenever their CTAs still fit in one wave: its
// chain of chunks per CTA halves, and each causal segment folds twice as many
// increments.
Plan plan_causal(int64_t BH, int nchunks, int sms, int D, bool gated) {
    Plan pl = plan_segments(BH, nchunks, sms);
    if (D == 64 && !gated && pl.nseg > 1 && pl.cps % 2 == 0 && pl.cps >= 4 && (int64_t)(pl.nseg - 1) * 2 * BH <= 2LL * sms)
        pl.sub = 2;
    return pl;
}

struct WsLayout {
    size_t S_seg = 0, Z_seg = 0, G_seg = 0, S_tot = 0, Z_tot = 0, total = 0;
};
// Causal with several segments: S_tot / Z_tot hold a copy of the initial
// state when the caller streams in place (S_out == S0), because the last
// segment writes the final state while other segments may still read S0.

WsLayout ws_layout(const Problem& P, bool causal, int nseg, int sub = 1) {
    WsLayout w;
    const size_t BH = static_cast<size_t>(P.B) * P.Hkv;
    const size_t D = P.Dk;
    size_t off = 0;
    if (causal && nseg <= 1) return w;
    // one increment per state-pass (sub-)segment
    const size_t ninc = static_cast<size_t>(nseg) * sub;
    w.S_seg = off;
    off += round_up(BH * ninc * D * D * sizeof(float));
    w.Z_seg = off;
    off += round_up(BH * ninc * D * sizeof(float));
    w.G_seg = off;
    off += round_up(BH * ninc * sizeof(float));
    {
        w.S_tot = off;
        off += round_up(BH * D * D * sizeof(float));
        w.Z_tot = off;
        off += round_up(BH * D * sizeof(float));
    }
    w.total = off;
    return w;
}

// Global state of the non-causal form: sum of the per-segment states in a
// fixed order (deterministic).
__global__ void segment_sum_kernel(const float* S_seg, const float* Z_seg, float* S_tot, float* Z_tot, int nseg,
                                   int D, int norm) {
    const int64_t bh = blockIdx.x;  // gridDim.x: up to 2^31 - 1 streams
    const int e = blockIdx.y * blockDim.x + threadIdx.x;
    const int DD = D * D;
    if (e < DD) {
        float acc = 0.f;
        for (int p = 0; p < nseg; ++p) acc += S_seg[(bh * nseg + p) * DD + e];
        S_tot[bh * DD + e] = acc;
    }
    if (norm && blockIdx.y == 0 && threadIdx.x < D) {
        float acc = 0.f;
        for (int p = 0; p < nseg; ++p) acc += Z_seg[(bh * nseg + p) * D + threadIdx.x];
        Z_tot[bh * D + threadIdx.x] = acc;
    }
}

// (D, H, T, B) view of an activation; loads use 64 x 64 boxes with the
// 128-byte swizzle, stores a plain (D, 1, 64, 1) box.
bool act_map(CUtensorMap* m, const void* base, int D, int H, int64_t T, int64_t B, bool store, bool f32) {
    const uint64_t es = f32 ? 4 : 2;
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)H, (uint64_t)T, (uint64_t)B};
    const uint64_t str[3] = {D * es, (uint64_t)H * D * es, (uint64_t)T * H * D * es};
    const uint32_t box_load[4] = {64, 1, 64, 1};
    const uint32_t box_store[4] = {(uint32_t)D, 1, 64, 1};
    return make_tensor_map(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, 4, dims,
                           str, store ? box_store : box_load,
                           store ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B);
}

cudaError_t run(const chunk::Launch& L, int D, cudaStream_t st) {
    if (L.args.mask) {  // the masked instantiations
        if (L.mode == chunk::kCausal) {
            if (D == 64) return L.out_bf16 ? chunk_run_causal_d64_bf16_mask(L, st) : chunk_run_causal_d64_f32_mask(L, st);
            return L.out_bf16 ? chunk_run_causal_d128_bf16_mask(L, st) : chunk_run_causal_d128_f32_mask(L, st);
        }
        return D == 64 ? chunk_run_other_d64_mask(L, st) : chunk_run_other_d128_mask(L, st);
    }
    if (L.mode == chunk::kCausal) {
        if (D == 64) return L.out_bf16 ? chunk_run_causal_d64_bf16(L, st) : chunk_run_causal_d64_f32(L, st);
        return L.out_bf16 ? chunk_run_causal_d128_bf16(L, st) : chunk_run_causal_d128_f32(L, st);
    }
    return D == 64 ? chunk_run_other_d64(L, st) : chunk_run_other_d128(L, st);
}

chunk::Launch base_launch(const Problem& P, int mode, const DevInfo& di) {
    chunk::Launch L;
    memset(&L, 0, sizeof(L));
    L.mode = mode;
    L.norm = P.norm != 0;
    L.gated = P.gated != 0;
    L.out_bf16 = P.out_bf16 != 0;
    chunk::Args& a = L.args;
    a.B = (int)P.B;
    a.T = (int)P.T;
    a.Hq = P.Hq;
    a.Hkv = P.Hkv;
    a.G = P.G;
    a.fmap = P.fmap;
    a.eps = P.eps;
    a.scale = P.scale;
    a.mask = P.mask;
    a.err = di.err;
    a.fold_r = 1;
    return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

uint64_t current_context_id() {
    using GetCurrent = PFN_cuCtxGetCurrent_v4000;
    using GetId = PFN_cuCtxGetId_v12000;
    static const std::pair<GetCurrent, GetId> fns = [] {
        void* a = nullptr;
        void* b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 4000, cudaEnableDefault, &qa) != cudaSuccess ||
            qa != cudaDriverEntryPointSuccess)
            a = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) != cudaSuccess ||
            qb != cudaDriverEntryPointSuccess)
            b = nullptr;
        return std::make_pair(reinterpret_cast<GetCurrent>(a), reinterpret_cast<GetId>(b));
    }();
    if (!fns.first || !fns.second) return 0;
    CUcontext c = nullptr;
    if (fns.first(&c) != CUDA_SUCCESS || !c) return 0;
    unsigned long long id = 0;
    if (fns.second(c, &id) != CUDA_SUCCESS) return 0;
    return static_cast<uint64_t>(id);
}

bool chunk_supported(const Problem& P) {
    if (!P.io_bf16 || P.Dk != P.Dv || (P.Dk != 64 && P.Dk != 128)) return false;
    if (P.T < 1 || P.T > 0x7fffffffLL - 64 || P.B > 0x7fffffffLL) return false;
    DevInfo di;
    return dev_info(&di);
}

bool chunk_pointers_ok(const void* q, const void* k, const void* v, const void* y) {
    return aligned16(q) && aligned16(k) && aligned16(v) && aligned16(y);
}

size_t chunk_workspace_bytes(const Problem& P, bool causal) {
    DevInfo di;
    if (!dev_info(&di)) return 0;
    const int nchunks = (int)((P.T + 63) / 64);
    if (causal) {
        const Plan pl = plan_causal((int64_t)P.B * P.Hkv, nchunks, di.sms, (int)P.Dk, P.gated != 0);
        return ws_layout(P, true, pl.nseg, pl.sub).total;
    }
    const Plan pl = plan_segments((int64_t)P.B * P.Hkv, nchunks, di.sms);
    return ws_layout(P, false, pl.nseg).total;
}

cudaError_t chunk_causal(const Problem& P, const void* q, const void* k, const void* v, const void* decay,
                         const float* S0, const float* Z0, void* y, float* S_out, float* Z_out, void* ws,
                         cudaStream_t st) {
    DevInfo di;
    if (!dev_info(&di)) return cudaErrorInvalidDevice;
    const int D = P.Dk;
    const int64_t BH = (int64_t)P.B * P.Hkv;
    const int nchunks = (int)((P.T + 63) / 64);
    const Plan pl = plan_causal(BH, nchunks, di.sms, D, P.gated != 0);
    const WsLayout wl = ws_layout(P, true, pl.nseg, pl.sub);
    char* w = static_cast<char*>(ws);

    chunk::Launch L = base_launch(P, chunk::kCausal, di);
    L.args.cps = pl.cps;
    L.args.nseg = pl.nseg;
    L.args.decay = static_cast<const __nv_bfloat16*>(decay);
    if (!act_map(&L.mq, q, D, P.Hq, P.T, P.B, false, false) || !act_map(&L.mk, k, D, P.Hkv, P.T, P.B, false, false) ||
        !act_map(&L.mv, v, D, P.Hkv, P.T, P.B, false, false))
        return cudaErrorInvalidValue;
    L.args.y = y;
    L.args.S_init = S0;
    L.args.Z_init = P.norm ? Z0 : nullptr;

    if (pl.nseg > 1) {
        float* S_seg = reinterpret_cast<float*>(w + wl.S_seg);
        float* Z_seg = reinterpret_cast<float*>(w + wl.Z_seg);
        float* G_seg = reinterpret_cast<float*>(w + wl.G_seg);
        cudaError_t e;
        if (S0 && S0 == S_out) {  // in-place streaming: read the initial state from a copy
            float* S_copy = reinterpret_cast<float*>(w + wl.S_tot);
            e = cudaMemcpyAsync(S_copy, S0, (size_t)BH * D * D * sizeof(float), cudaMemcpyDeviceToDevice, st);
            if (e != cudaSuccess) return e;
            L.args.S_init = S_copy;
        }
        if (P.norm && Z0 && Z0 == Z_out) {
            float* Z_copy = reinterpret_cast<float*>(w + wl.Z_tot);
            e = cudaMemcpyAsync(Z_copy, Z0, (size_t)BH * D * sizeof(float), cudaMemcpyDeviceToDevice, st);
            if (e != cudaSuccess) return e;
            L.args.Z_init = Z_copy;
        }
        // the state pass over segments 0..nseg-2, each as pl.sub sub-segments
        chunk::Launch Ls = L;
        Ls.mode = chunk::kState;
        Ls.args.cps = pl.cps / pl.sub;
        Ls.args.nseg = pl.nseg * pl.sub;
        Ls.grid = dim3((unsigned)BH, (unsigned)((pl.nseg - 1) * pl.sub));
        Ls.args.S_dst = S_seg;
        Ls.args.Z_dst = P.norm ? Z_seg : nullptr;
        Ls.args.G_dst = G_seg;
        e = run(Ls, D, st);
        if (e != cudaSuccess) return e;
        L.args.S_seg = S_seg;
        L.args.Z_seg = P.norm ? Z_seg : nullptr;
        L.args.G_seg = G_seg;
        L.args.fold_r = pl.sub;
        L.pdl = true;  // overlaps the state pass's tail; waits for it before the fold
    }
    L.grid = dim3((unsigned)BH, (unsigned)pl.nseg);
    L.args.S_dst = S_out;
    L.args.Z_dst = P.norm ? Z_out : nullptr;
    return run(L, D, st);
}

cudaError_t chunk_noncausal(const Problem& P, const void* q, const void* k, const void* v, void* y, void* ws,
                            cudaStream_t st) {
    DevInfo di;
    if (!dev_info(&di)) return cudaErrorInvalidDevice;
    const int D = P.Dk;
    const int64_t BH = (int64_t)P.B * P.Hkv;
    const int nchunks = (int)((P.T + 63) / 64);
    const Plan pl = plan_segments(BH, nchunks, di.sms);
    const WsLayout wl = ws_layout(P, false, pl.nseg);
    char* w = static_cast<char*>(ws);
    float* S_seg = reinterpret_cast<float*>(w + wl.S_seg);
    float* Z_seg = reinterpret_cast<float*>(w + wl.Z_seg);
    float* S_tot = reinterpret_cast<float*>(w + wl.S_tot);
    float* Z_tot = reinterpret_cast<float*>(w + wl.Z_tot);

    chunk::Launch L = base_launch(P, chunk::kState, di);
    L.gated = false;
    L.args.cps = pl.cps;
    L.args.nseg = pl.nseg;
    if (!act_map(&L.mq, q, D, P.Hq, P.T, P.B, false, false) || !act_map(&L.mk, k, D, P.Hkv, P.T, P.B, false, false) ||
        !act_map(&L.mv, v, D, P.Hkv, P.T, P.B, false, false))
        return cudaErrorInvalidValue;
    L.args.y = y;
    L.grid = dim3((unsigned)BH, (unsigned)pl.nseg);
    L.args.S_dst = S_seg;
    L.args.Z_dst = P.norm ? Z_seg : nullptr;
    cudaError_t e = run(L, D, st);
    if (e != cudaSuccess) return e;
    const int DD = D * D;
    segment_sum_kernel<<<dim3((unsigned)BH, (DD + 255) / 256), 256, 0, st>>>(S_seg, Z_seg, S_tot, Z_tot, pl.nseg, D,
                                                                           P.norm);
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    chunk::Launch La = L;
    La.mode = chunk::kApply;
    La.args.S_init = S_tot;
    La.args.Z_init = P.norm ? Z_tot : nullptr;
    La.args.S_dst = nullptr;
    La.args.Z_dst = nullptr;
    La.grid = dim3((unsigned)BH, (unsigned)pl.nseg);
    return run(La, D, st);
}

int device_sm_count() {
    DevInfo di;
    return dev_info(&di) ? di.sms : 0;
}

unsigned* device_error_word() {
    DevInfo di;
    return dev_info(&di) ? di.err : nullptr;
}

unsigned chunk_device_error(bool reset) {
    DevInfo di;
    if (!dev_info(&di)) return 0;
    unsigned v = 0;
    if (cudaMemcpy(&v, di.err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return ~0u;
    if (reset && v) {
        unsigned z = 0;
        cudaMemcpy(di.err, &z, sizeof(z), cudaMemcpyHostToDevice);
    }
    return v;
}

}  // namespace la
