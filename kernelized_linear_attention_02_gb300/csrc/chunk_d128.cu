// chunk_d128.cu -- tensor-core chunk kernel, head size 128.
#include "chunk_launch.cuh"

namespace la {
cudaError_t chunk_run_d128(const chunk::Launch& L, cudaStream_t st) { return chunk::run_d<128>(L, st); }
}  // namespace la

#ifdef LA_TRACE
LA_TRACE_DUMP(la_trace_dump_d128)
#endif
