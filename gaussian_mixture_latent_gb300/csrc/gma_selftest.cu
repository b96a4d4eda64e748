// Self-test of the device-side failure path: a bounded wait that runs out.
//
// Every mbarrier wait in the library's kernels gives up after one second on the
// global nanosecond timer, raises its CTA's abort flag and posts GMA_ERR_TIMEOUT to the
// status word at the start of the workspace.  selftest_timeout_kernel waits, with
// that same bounded wait, on a barrier that nothing arrives at, so the path can be
// exercised without faulting or hanging the GPU: the kernel ends after the bound.
#include "gma_internal.h"
#include "gma_sm100.cuh"

namespace gma {
namespace {

__global__ void selftest_timeout_kernel(unsigned *status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ volatile int flag;
    if (threadIdx.x == 0) {
        sm100::mbar_init(&bar, 1);
        flag = 0;
        sm100::fence_mbar_init();
    }
    __syncthreads();
    const sm100::Abort ab{&flag, status};
    (void)sm100::mbar_wait(&bar, 0, ab, kDevErrTimeout);      // phase 0 never completes
}

}  // namespace

cudaError_t selftest_timeout(void *ws, cudaStream_t s) {
    selftest_timeout_kernel<<<1, 32, 0, s>>>(static_cast<unsigned *>(ws));
    return cudaGetLastError();
}

}  // namespace gma
