// Bulk-copy (TMA, 1-D) and mbarrier helpers for sm_90+ / sm_103a, as inline PTX.
//
// A stage of a pipeline is filled by cp.async.bulk copies from global memory into shared
// memory; an mbarrier counts the bytes as they land. Every wait on an mbarrier is
// bounded: past the limit the waiter records a status code in global memory and gives
// up, so a copy that never completes cannot hang the GPU.
#pragma once

#include <stdint.h>

namespace ob {

// Status codes a kernel may leave in its status word (0 = fine).
constexpr unsigned kStatusWaitTimeout = 1u;

// Longest a warp waits for one pipeline stage before giving up: 2 s of GPU time.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t arrivals)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(arrivals) : "memory");
}

// Make barrier initialisation visible to the bulk-copy (async) proxy.
__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// One arrival that also announces `bytes` of copies still to land in this phase.
__device__ __forceinline__ void mbar_arrive_expect(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete, at most limit_ns (and at most
// 2^30 polls). Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t spins = 0; spins < (1u << 30); ++spins) {
        if (mbar_test(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
    return false;
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity)
{
    return mbar_wait_for(bar, parity, kWaitLimitNs);
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from global to
// this CTA's shared memory, completing on mbarrier `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// The same with an L2 eviction-priority hint (for data read exactly once).
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void bulk_load_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                               uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}

// Per-thread asynchronous copies of 16 bytes from global to shared memory (both addresses
// 16-byte aligned), grouped by commit and awaited by count: a copy lands in shared memory
// without passing through registers, so a warp can keep several stages in flight at no
// register cost. The wait is a hardware wait for this thread's own copies (no polling);
// other lanes see the data after a __syncwarp.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint64_t pol)
{
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's committed groups are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Programmatic dependent launch (sm_90+). A kernel launched with the programmatic
// stream-serialization attribute may start while the kernel before it on the stream is
// still running; pdl_wait() blocks until that kernel has completed and its writes are
// visible (it returns at once when there is no such kernel), so it comes before the
// kernel's first global-memory access, read or write. pdl_allow_next() lets the kernel
// after this one be scheduled (its blocks then wait in their own pdl_wait()); since every
// kernel of the chain waits before touching memory, each one also follows all earlier
// ones.
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void pdl_allow_next()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace ob
