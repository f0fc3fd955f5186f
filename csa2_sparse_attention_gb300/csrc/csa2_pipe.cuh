// mbarrier and bulk-copy helpers for the producer/consumer pipelines.  Every
// wait is bounded in time (globaltimer) so a kernel can never spin forever:
// a wait that gives up returns false and the caller records
// CSA2_ERR_TIMEOUT and leaves.
#pragma once

#include <cstdint>

namespace csa2 {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// make barrier initialization visible to the async (bulk copy) proxy
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;\nfence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// One test of the phase; the thread may be suspended until the phase
// completes, for at most about `suspend_ns` nanoseconds, so waiting warps do
// not take issue slots from the working ones.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity, uint32_t suspend_ns = 1000000u) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(suspend_ns)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits that drain copies and MMAs already issued after a give-up use their
// own limit, which the test hook (csa2_debug_wait_limit) does not shorten.
constexpr uint64_t kDrainNs = 100000000ull;

// Wait for the completion of the barrier phase with the given parity; gives
// up after about `limit_ns` nanoseconds.  Kernels take the limit as a launch
// argument: 2 s, unless a test of the give-up paths passes a limit under
// 1 ms, which makes every such wait give up at once.  (Any second wait form
// in the loop -- a polling test_wait, even predicated off -- slowed the
// decode scan by 7%, so the test form only masks the result.)
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    const bool give_up = limit_ns < 1000000u;
    if (mbar_try_wait(bar, parity) & !give_up) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (give_up | (global_ns() - t0 > limit_ns)) return false;
        if (mbar_try_wait(bar, parity)) return true;
    }
}

// One bulk copy global -> shared memory that completes `bytes` of the
// barrier's transaction count (both addresses 16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// One TMA gather: four one-row boxes of a 2-D tensor map (rows r0..r3, from
// column 0) into consecutive box-sized slots at dst, completing their bytes
// on the barrier.  dst 128-byte aligned; the map lives in kernel parameter
// space (__grid_constant__).
__device__ __forceinline__ void tma_gather4(void* dst, const void* tmap, int r0, int r1, int r2, int r3,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
        : "memory");
}

}  // namespace csa2
