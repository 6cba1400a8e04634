// Self-test of the bounded-wait path every kernel of the library relies on:
// one CTA waits on an mbarrier that nothing ever completes, with the same
// bounded try_wait loop as the kernels but a caller-chosen limit, and reports
// KDA_DEV_TIMEOUT through the device status word when the wait gives up. The
// GPU is never hung: the wait ends after `limit` SM clocks whatever happens.
#include "kda_internal.cuh"
#include "sm100_ptx.cuh"

namespace kda {
namespace {

__global__ void kda_selftest_wait_kernel(long long limit, int* d_status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        ptx::fence_mbarrier_init();
    }
    __syncthreads();
    const bool ok = ptx::mbar_wait(&bar, 0, limit);  // no arrive is ever issued
    report_flags(d_status, ok ? 0 : KDA_DEV_TIMEOUT);
}

}  // namespace

cudaError_t launch_selftest_wait(long long limit, int* d_status, cudaStream_t stream) {
    kda_selftest_wait_kernel<<<1, 32, 0, stream>>>(limit, d_status);
    return cudaGetLastError();
}

}  // namespace kda
