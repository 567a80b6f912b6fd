// Pieces shared by the tcgen05 kernels: bounded mbarrier waits with a CTA
// abort flag, and the TMA tensor-map encoder for bf16 [units][rows][d] views.
#pragma once

#include <cudaTypedefs.h>

#include "statekv_internal.cuh"
#include "sm100_ptx.cuh"

namespace statekv {

constexpr uint64_t kTimeoutNs = 1000000000ull;   // 1 s per wait

struct Sync {
    uint32_t bar0;                 // smem address of barrier 0
    volatile uint32_t* abort;      // CTA-wide abort flag (smem)
    uint32_t* err;

    __device__ uint32_t bar(int i) const { return bar0 + 8u * (uint32_t)i; }

    // Wait for the phase of the given parity; gives up on abort or timeout.
    // After one non-blocking probe the thread sleeps in try_wait, which
    // returns as soon as the phase completes (a spin that also reads the
    // global timer reacts hundreds of cycles late).
    __device__ bool wait(int i, uint32_t parity, uint32_t site) const {
        const uint32_t b = bar(i);
        if (ptx::mbar_poll(b, parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        for (;;) {
            if (ptx::mbar_wait_hint(b, parity, 20000u)) return true;
            if (*abort) return false;
            if (globaltimer_ns() - t0 > kTimeoutNs) {
                *abort = 1u;
                record_error(err, (uint32_t)STATEKV_E_TIMEOUT, site, (uint32_t)i);
                return false;
            }
        }
    }
    // wait() for a barrier that the other CTA of a cluster arrives on after
    // writing into this CTA's shared memory (acquire at cluster scope)
    __device__ bool wait_cluster(int i, uint32_t parity, uint32_t site) const {
        const uint32_t b = bar(i);
        if (ptx::mbar_poll_cluster(b, parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        for (;;) {
            if (ptx::mbar_wait_hint_cluster(b, parity, 20000u)) return true;
            if (*abort) return false;
            if (globaltimer_ns() - t0 > kTimeoutNs) {
                *abort = 1u;
                record_error(err, (uint32_t)STATEKV_E_TIMEOUT, site, (uint32_t)i);
                return false;
            }
        }
    }
    // Teardown wait: ignores the abort flag, still bounded.
    __device__ void drain(int i, uint32_t parity) const {
        const uint32_t b = bar(i);
        const uint64_t t0 = globaltimer_ns();
        while (!ptx::mbar_wait_hint(b, parity, 20000u)) {
            if (globaltimer_ns() - t0 > kTimeoutNs) {
                record_error(err, (uint32_t)STATEKV_E_TIMEOUT, kSiteDrain, (uint32_t)i);
                return;
            }
        }
    }
};


// 3-D bf16 view [units][rows][d] read in boxes of 64 columns (one 128-byte
// swizzle row) x box_rows rows; rows past `rows` read as zero.
bool encode_view(CUtensorMap* m, const void* base, int d, int64_t rows, int64_t units,
                 int box_rows);

}  // namespace statekv
