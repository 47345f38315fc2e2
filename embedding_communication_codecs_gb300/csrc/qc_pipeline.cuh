// qc_pipeline.cuh -- multi-stage shared-memory pipeline fed by the Tensor Memory
// Accelerator's bulk copies (cp.async.bulk, 1-D), with mbarrier completion.
//
// One thread of a block issues the bulk copies of a tile into a stage and arms
// the stage's mbarrier with the byte count; every consumer thread waits on the
// barrier's phase before reading the stage.  Small per-bucket metadata that has
// no 16-byte alignment guarantee is fetched with 4-byte cp.async copies whose
// completion is tracked on the same barrier (cp.async.mbarrier.arrive.noinc).
//
// Every wait is bounded in time: a wait that has not completed after
// kWaitNs nanoseconds of the GPU's global timer (or, as a backstop should that
// timer not advance, after kWaitRoundsBackstop tries) gives up and reports
// failure; the block stops at its next agreement point, and the kernel records
// the failure in a device flag that the host reads with
// qc_take_device_errors(), and in the caller's status word if one was set
// (qc_set_status_word).  Nothing spins forever.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace qc {

// A stalled pipeline gives up after 2 s.  An unsuccessful try_wait may return
// early or late (the suspend time is the implementation's choice, the hint
// below only a suggestion), so the limit is kept on the global timer and on the
// SM's cycle counter; the round count is only a backstop.
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kWaitRoundsBackstop = 1u << 26;

// Named barrier 1 over the first `threads` threads of the block (the consumer
// warps of a warp-specialised block; the producer warp never takes part).
template <int THREADS>
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(THREADS) : "memory");
}

// The same barrier, returning whether `v` holds on every participating thread.
template <int THREADS>
__device__ __forceinline__ bool consumer_sync_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "n"(THREADS)
        : "memory");
    return r != 0u;
}
constexpr uint32_t kErrPipelineTimeout = 1u;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Makes barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier shared-memory accesses (generic proxy) before the
// bulk copies it issues next (async proxy).
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from
// global memory into this block's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 4-byte asynchronous copy global -> shared (no alignment beyond 4 bytes).
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}

// 16-byte asynchronous copy global -> shared (both addresses 16-byte aligned),
// cached in L2 only; completion by cp_async_wait_all() of the issuing thread.
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}

// Arrive on `bar` once this thread's earlier cp.async copies have landed (the
// arrival is one of the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// One try with a suspend-time hint: the thread sleeps in the barrier unit until
// the phase completes or about kTryWaitHintNs pass, instead of spinning on
// issue slots that the block's working warps need.
constexpr uint32_t kTryWaitHintNs = 1000000u;

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kTryWaitHintNs)
        : "memory");
    return done != 0;
}

// The GPU's global timer, in nanoseconds.
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity for at most about limit_ns
// nanoseconds (the timer is read after every unsuccessful try); false if it
// never completed.
// The SM's cycle counter bounds the wait as well (4 cycles per nanosecond of
// the limit: about twice the limit at the highest clock), and so does a count
// of tries, so that no single clock has to be trusted.
__device__ __forceinline__ bool mbar_wait_ns(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    const long long c0 = clock64();
    const long long cycle_limit = static_cast<long long>(4u * limit_ns + (1u << 20));
    for (uint32_t r = 1; r < kWaitRoundsBackstop; ++r) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns || clock64() - c0 > cycle_limit) return false;
    }
    return false;
}

// The pipelines' bounded wait.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    return mbar_wait_ns(bar, parity, kWaitNs);
}

// Records failure bits in a translation unit's device flag and, if the launch
// carries one, in the caller's status word.
__device__ __forceinline__ void report_failure(unsigned int *flag, uint32_t *status, uint32_t bits) {
    atomicOr(flag, bits);
    if (status) atomicOr(status, bits);
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__host__ __device__ constexpr uint32_t floor16(uint64_t bytes) {
    return static_cast<uint32_t>(bytes & ~static_cast<uint64_t>(15));
}

// Defines FN (cudaError_t FN(uint32_t *flags)): stores FLAG's value in *flags
// and clears it in one atomic exchange on the device (a one-thread kernel on the
// legacy stream, then a copy of the exchanged value), so a bit that a kernel
// sets at any moment is reported exactly once.  For use at namespace qc scope.
#define QC_DEFINE_TAKE_FLAG(FN, FLAG)                                               \
    static __device__ unsigned int FLAG##_taken;                                    \
    static __global__ void FLAG##_exchange() { FLAG##_taken = atomicExch(&FLAG, 0u); } \
    cudaError_t FN(uint32_t *flags) {                                               \
        *flags = 0u;                                                                \
        FLAG##_exchange<<<1, 1>>>();                                                \
        cudaError_t e = cudaGetLastError();                                         \
        if (e != cudaSuccess) return e;                                             \
        unsigned int v = 0u;                                                        \
        e = cudaMemcpyFromSymbol(&v, FLAG##_taken, sizeof v);                       \
        *flags = v;                                                                 \
        return e;                                                                   \
    }

}  // namespace qc
