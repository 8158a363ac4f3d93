// chunk_launch.cuh -- instantiates the tensor-core chunk kernel for one head
// size D and one group of modes (included by chunk_d{64,128}_{causal,other}.cu,
// so the variants compile in parallel translation units).
#pragma once

#include <atomic>

#include "chunk.cuh"
#include "kernels.h"

namespace la {
namespace chunk {

template <int D, int MODE, bool NORM, int FMAP, bool GATED, bool OUTBF, int SPLIT = 0, bool MASK = false>
cudaError_t run_one(const Launch& L, cudaStream_t st) {
    using Cf = Cfg<D, MODE, NORM, FMAP, GATED, OUTBF, SPLIT == 2>;
    auto kern = chunk_kernel<D, MODE, NORM, FMAP, GATED, OUTBF, SPLIT, MASK>;
    // per device: the context in which the shared-memory limit of this
    // instantiation was raised (0 = not yet); a new context (a device reset)
    // raises it again.  Two threads may both raise it: the call is idempotent.
    static std::atomic<uint64_t> configured[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    const uint64_t ctx = current_context_id();
    if (ctx == 0 || configured[dev].load(std::memory_order_acquire) != ctx) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::kSmem);
        if (e != cudaSuccess) return e;
        configured[dev].store(current_context_id(), std::memory_order_release);
    }
    if (L.pdl) {
        // may start while the previous kernel (the segment state pass) drains;
        // the kernel waits for it (griddepcontrol.wait) before reading its output
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = L.grid;
        cfg.blockDim = dim3(block_threads<Cf::kSplitMma && SPLIT != 0>());
        cfg.dynamicSmemBytes = Cf::kSmem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, L.args, L.mq, L.mk, L.mv);
        if (e != cudaSuccess) return e;
    } else {
        kern<<<L.grid, block_threads<Cf::kSplitMma && SPLIT != 0>(), Cf::kSmem, st>>>(L.args, L.mq, L.mk, L.mv);
    }
    note_launch();
    return cudaGetLastError();
}

// OUT: 1 = bf16 output, 0 = float32 output (the state pass writes no output);
// MASK: the instantiations that read a sequence-validity mask
template <int D, int MODE, int OUT, bool MASK = false>
struct Dispatch {
    template <bool NORM, int FMAP, bool GATED>
    static cudaError_t one(const Launch& L, cudaStream_t st) {
        // linear causal rule: the two-issuer kernel for grouped query heads, and
        // at head size 128 with one query head per kv head (at head size 64 the
        // single issuer measured faster there)
        if constexpr (MODE == kCausal && !GATED) {
            if (L.args.G > 1) return run_one<D, MODE, NORM, FMAP, GATED, OUT == 1, 2, MASK>(L, st);
            if constexpr (D == 128) return run_one<D, MODE, NORM, FMAP, GATED, OUT == 1, 1, MASK>(L, st);
        }
        return run_one<D, MODE, NORM, FMAP, GATED, OUT == 1, 0, MASK>(L, st);
    }
    template <bool NORM>
    static cudaError_t fmap(const Launch& L, cudaStream_t st) {
        switch (L.args.fmap) {
        case LA_FMAP_ELU_PLUS_ONE: return one<NORM, LA_FMAP_ELU_PLUS_ONE, false>(L, st);
        case LA_FMAP_RELU_EPS: return one<NORM, LA_FMAP_RELU_EPS, false>(L, st);
        default: return one<NORM, LA_FMAP_NONE, false>(L, st);
        }
    }
    static cudaError_t run(const Launch& L, cudaStream_t st) {
        // the gated rule is defined without a feature map or normalizer
        if (MODE != kApply && L.gated) return one<false, LA_FMAP_NONE, true>(L, st);
        return L.norm ? fmap<true>(L, st) : fmap<false>(L, st);
    }
};

}  // namespace chunk
}  // namespace la
