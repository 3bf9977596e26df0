// selftest.cu -- device self-test of the bounded waits.
//
// Every wait of the library's kernels on an mbarrier gives up after
// NA_WAIT_LIMIT_CYCLES (2^31 SM cycles, about a second) and reports
// NA_ERR_DEVICE_TIMEOUT in the caller's status word instead of hanging the
// GPU.  This entry point runs that same wait on a barrier that no thread ever
// arrives on, so a test can watch the limit run out and the status come back
// while the context stays usable.  Nothing faults: the wait simply ends.
#include "na_internal.cuh"

namespace {

__global__ void wait_timeout_kernel(int32_t *status)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0)
        mbar_init(&bar, 1);  // phase 0 completes after one arrival, which never comes
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait_bounded(&bar, 0))
        na_report(status, NA_ERR_DEVICE_TIMEOUT);
    __syncthreads();
}

}  // namespace

extern "C" int na_selftest_wait_timeout(int32_t *status, void *stream)
{
    if (!status)
        return NA_ERR_INVALID_ARG;
    wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status);
    return cudaGetLastError() == cudaSuccess ? NA_OK : NA_ERR_CUDA;
}
