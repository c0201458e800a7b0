// wait.cuh -- bounded barrier waits.  A wait that runs past its budget records
// a timeout in the device status word and returns false; the caller then
// stops issuing work and goes to the kernel's teardown, which still releases
// TMEM.  No wait in these kernels is unbounded.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace gemm_gb300 {

// Status word layout: bits 0-7 the gemm_status_t code, bits 8-15 the wait
// site, bits 16-31 the low bits of the CTA index.
constexpr uint32_t kStatusTimeout = 5;

enum WaitSite : uint32_t {
    kSiteProducerEmpty = 1,
    kSiteProducerTail = 2,
    kSiteMmaTmemEmpty = 3,
    kSiteMmaFull = 4,
    kSiteMmaDrain = 5,
    kSiteEpilogueTmemFull = 6,
    kSiteSplitPieces = 7,
    kSiteSelfTest = 8,
};

__device__ __forceinline__ void record_timeout(uint32_t* status, uint32_t site) {
    atomicCAS(status, 0u, kStatusTimeout | (site << 8) | ((blockIdx.x & 0xFFFFu) << 16));
}

// Wait for the phase of parity `parity` of `bar` to complete, for at most
// `timeout_ns` of wall-clock time.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, uint32_t* status,
                                           uint32_t site, uint64_t timeout_ns) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (ptx::mbar_try_wait(bar, parity)) return true;
        if (ptx::globaltimer_ns() - t0 > timeout_ns) {
            record_timeout(status, site);
            return false;
        }
    }
}

// Wait until the global counter reaches `target` (other CTAs of the same
// launch increment it), for at most `timeout_ns`.  Only used between CTAs that
// are resident at the same time (the planner guarantees it).
__device__ __forceinline__ bool wait_count(const uint32_t* addr, uint32_t target, uint32_t* status,
                                           uint32_t site, uint64_t timeout_ns) {
    uint64_t t0 = 0;
    while (true) {
        uint32_t v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
        if (v >= target) return true;
        const uint64_t now = ptx::globaltimer_ns();
        if (t0 == 0) {
            t0 = now;
        } else if (now - t0 > timeout_ns) {
            record_timeout(status, site);
            return false;
        }
        __nanosleep(64);
    }
}

// Every lane of the warp waits; the result is made uniform across the warp
// (false if any lane gave up) so later .sync.aligned instructions stay
// convergent.
__device__ __forceinline__ bool wait_phase_warp(uint32_t bar, uint32_t parity, uint32_t* status,
                                                uint32_t site, uint64_t timeout_ns) {
    const bool ok = wait_phase(bar, parity, status, site, timeout_ns);
    return __all_sync(0xffffffffu, ok) != 0;
}

}  // namespace gemm_gb300
