// selftest.cu -- failure-path check of the bounded pipeline waits.
//
// Every wait of the tensor-core kernels (umma.cuh: mbar_wait, warp_wait)
// gives up after a time limit, records a bit in the device error word and
// lets the kernel return, instead of hanging the GPU.  This kernel runs both
// wait forms on an mbarrier that nothing ever arrives at, with a short
// limit, so that the give-up path runs for real: it holds no tensor memory
// and has no copy or tensor-core operation in flight, so returning early is
// always clean.
#include "kernels.h"
#include "umma.cuh"

namespace la {
namespace {

__global__ void bounded_wait_selftest_kernel(unsigned* err, uint64_t limit_ns) {
    __shared__ uint64_t never;  // no thread ever arrives on it
    if (threadIdx.x == 0) {
        umma::mbar_init(&never, 1);
        umma::fence_barrier_init();
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    if (warp == 0) {
        // warp-uniform form: all lanes poll, lane 0 decides and reports
        umma::warp_wait(&never, 0, err, LA_SELFTEST_WARP_WAIT, limit_ns);
    } else if (warp == 1 && (threadIdx.x & 31) == 0) {
        // single-thread form
        umma::mbar_wait(&never, 0, err, LA_SELFTEST_THREAD_WAIT, limit_ns);
    }
    __syncthreads();
}

}  // namespace

cudaError_t bounded_wait_selftest(uint32_t limit_us, cudaStream_t st) {
    unsigned* err = device_error_word();
    if (!err) return cudaErrorInvalidDevice;
    bounded_wait_selftest_kernel<<<1, 64, 0, st>>>(err, (uint64_t)limit_us * 1000ull);
    note_launch();
    return cudaGetLastError();
}

}  // namespace la
