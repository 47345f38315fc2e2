// qc_selftest.cu -- self-test of the pipelines' failure path.  One block waits
// on an mbarrier that nothing ever arrives at, with the same bounded wait the
// pipelined kernels use but a caller-chosen number of tries; the wait runs out
// and the block records the pipeline-timeout flag, exactly as a stalled
// pipeline would, then returns.  No fault, no trap: the context stays usable.
#include "qc_device.cuh"
#include "qc_internal.h"
#include "qc_pipeline.cuh"

namespace qc {

static __device__ unsigned int g_selftest_errors;

namespace {

__global__ void wait_timeout_kernel(uint32_t rounds) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // one arrival would complete phase 0; none comes
        fence_barrier_init();
    }
    __syncthreads();
    const bool ok = mbar_wait_rounds(&bar, 0u, rounds);
    if (!__all_sync(kFull, ok) && threadIdx.x == 0) atomicOr(&g_selftest_errors, kErrPipelineTimeout);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(uint32_t rounds, cudaStream_t stream) {
    wait_timeout_kernel<<<1, 32, 0, stream>>>(rounds);
    return cudaGetLastError();
}

uint32_t take_selftest_errors() {
    unsigned int v = 0, zero = 0;
    cudaMemcpyFromSymbol(&v, g_selftest_errors, sizeof v);
    cudaMemcpyToSymbol(g_selftest_errors, &zero, sizeof zero);
    return v;
}

}  // namespace qc
