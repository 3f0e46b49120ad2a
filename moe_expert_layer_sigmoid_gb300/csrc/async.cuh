// mbarrier and bulk-copy helpers shared by the kernels that stage data with
// the TMA unit (cp.async.bulk) or wait on mbarriers.  Every wait is bounded:
// it gives up after kWaitNs, records kErrWaitTimeout in the workspace header
// and raises the CTA's abort flag, so a broken pipeline ends the kernel with
// an error status instead of hanging the GPU.
#pragma once

#include "common.cuh"

namespace moe {

constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s: a wait that long means something broke

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 1000000;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// The wait limit: the header's test setting, else kWaitNs.
__device__ __forceinline__ uint64_t wait_limit(const WsHeader* hdr) {
    const uint64_t v = hdr ? *reinterpret_cast<const volatile uint64_t*>(&hdr->wait_ns) : 0;
    return v ? v : kWaitNs;
}

// Bounded wait: gives up after the wait limit (or once another warp gave up),
// records the failure in the workspace header and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          WsHeader* hdr) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    const uint64_t limit = wait_limit(hdr);
    for (uint32_t i = 1;; ++i) {
        if (mbar_try(bar, parity)) return true;
        if ((i & 255u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > limit) {
                *abort_flag = 1;
                record_error(hdr, kErrWaitTimeout);
                return false;
            }
        }
    }
}

// Teardown wait for this thread's own asynchronous work (copies or MMAs it
// issued) after an abort: ignores the abort flag, still bounded by the limit.
__device__ __forceinline__ bool mbar_drain(uint32_t bar, uint32_t parity, WsHeader* hdr) {
    const uint64_t t0 = globaltimer();
    const uint64_t limit = wait_limit(hdr);
    for (uint32_t i = 0;; ++i) {
        if (mbar_try(bar, parity)) return true;
        if ((i & 255u) == 255u && globaltimer() - t0 > limit) {
            record_error(hdr, kErrWaitTimeout);
            return false;
        }
    }
}

// Plain bulk copy global -> shared, completion counted on the mbarrier (bytes).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

}  // namespace moe
