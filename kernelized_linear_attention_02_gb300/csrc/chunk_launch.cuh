// chunk_launch.cuh -- instantiates the tensor-core chunk kernel for one head
// size D (included by chunk_d64.cu and chunk_d128.cu, so the two sizes
// compile in parallel).
#pragma once

#include "chunk.cuh"
#include "kernels.h"

namespace la {
namespace chunk {

template <int D, int MODE, bool NORM, bool SPLITK, bool GATED, bool OUTBF>
cudaError_t run_one(const Launch& L, cudaStream_t st) {
    using Cf = Cfg<D, MODE, NORM, SPLITK, GATED, OUTBF>;
    auto kern = chunk_kernel<D, MODE, NORM, SPLITK, GATED, OUTBF>;
    static int configured = -1;  // device on which the shared-memory limit was raised
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured != dev) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::kSmem);
        if (e != cudaSuccess) return e;
        configured = dev;
    }
    kern<<<L.grid, kThreads, Cf::kSmem, st>>>(L.args, L.mq, L.mk, L.mv);
    note_launch();
    return cudaGetLastError();
}

template <int D, int MODE, bool NORM, bool SPLITK, bool GATED>
cudaError_t run_out(const Launch& L, cudaStream_t st) {
    if (MODE == kState) return run_one<D, MODE, NORM, SPLITK, GATED, true>(L, st);
    return L.out_bf16 ? run_one<D, MODE, NORM, SPLITK, GATED, true>(L, st)
                      : run_one<D, MODE, NORM, SPLITK, GATED, false>(L, st);
}

template <int D, int MODE>
cudaError_t run_mode(const Launch& L, cudaStream_t st) {
    if (MODE == kApply) {
        return L.norm ? run_out<D, MODE, true, false, false>(L, st) : run_out<D, MODE, false, false, false>(L, st);
    }
    if (L.gated) return run_out<D, MODE, false, true, true>(L, st);
    if (L.norm)
        return L.splitk ? run_out<D, MODE, true, true, false>(L, st) : run_out<D, MODE, true, false, false>(L, st);
    return L.splitk ? run_out<D, MODE, false, true, false>(L, st) : run_out<D, MODE, false, false, false>(L, st);
}

template <int D>
cudaError_t run_d(const Launch& L, cudaStream_t st) {
    switch (L.mode) {
    case kCausal: return run_mode<D, kCausal>(L, st);
    case kState: return run_mode<D, kState>(L, st);
    default: return run_mode<D, kApply>(L, st);
    }
}

}  // namespace chunk
}  // namespace la

#ifdef LA_TRACE
// Trace builds only: copy out (and reset) this unit's event buffer.
#define LA_TRACE_DUMP(NAME)                                                                              \
    extern "C" int NAME(unsigned* count, unsigned long long* times, unsigned* tags) {                   \
        using namespace la::trace;                                                                      \
        if (cudaDeviceSynchronize() != cudaSuccess) return -1;                                          \
        cudaMemcpyFromSymbol(count, g_count, sizeof(unsigned) * kTraceCtas);                            \
        cudaMemcpyFromSymbol(times, g_time, sizeof(unsigned long long) * kTraceCtas * kTraceEvents);    \
        cudaMemcpyFromSymbol(tags, g_tag, sizeof(unsigned) * kTraceCtas * kTraceEvents);                \
        unsigned long long zt[kTraceEvents] = {};                                                        \
        for (int c = 0; c < kTraceCtas; ++c)                                                             \
            cudaMemcpyToSymbol(g_time, zt, sizeof(zt), sizeof(zt) * c);                                  \
        return 0;                                                                                       \
    }
#endif
