// qc_selftest.cu -- self-test of the pipelines' failure path.  One block waits
// on an mbarrier that nothing ever arrives at, with the same time-bounded wait
// the pipelined kernels use but a caller-chosen limit; the wait runs out and the
// block records the pipeline-timeout flag (and the caller's status word, if
// set), exactly as a stalled pipeline would, then returns.  No fault, no trap: the context stays usable.
#include "qc_device.cuh"
#include "qc_internal.h"
#include "qc_pipeline.cuh"

namespace qc {

static __device__ unsigned int g_selftest_errors;

namespace {

__global__ void wait_timeout_kernel(uint64_t limit_ns, uint32_t *status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // one arrival would complete phase 0; none comes
        fence_barrier_init();
    }
    __syncthreads();
    const bool ok = mbar_wait_ns(&bar, 0u, limit_ns);
    if (!__all_sync(kFull, ok) && threadIdx.x == 0)
        report_failure(&g_selftest_errors, status, kErrPipelineTimeout);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(uint32_t timeout_us, uint32_t *status, cudaStream_t stream) {
    wait_timeout_kernel<<<1, 32, 0, stream>>>(static_cast<uint64_t>(timeout_us) * 1000u, status);
    return cudaGetLastError();
}

QC_DEFINE_TAKE_FLAG(take_selftest_errors, g_selftest_errors)

}  // namespace qc
