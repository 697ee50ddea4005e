// sb_pipe.cuh -- the time-bounded mbarrier waits shared by the pipelined kernels.
//
// Every wait polls with mbarrier.try_wait and gives up after a %globaltimer limit: it then
// records SB_ERR_DEVICE_TIMEOUT (tagged with the launch epoch) in the caller-visible status
// word and raises a CTA-wide abort flag that the other roles' waits notice.
#pragma once
#include <cstdint>

#include "sb_ptx.cuh"

namespace sb {

struct WaitCtx {
    unsigned long long *status;  // (epoch << 32) | code, updated with record_status
    uint32_t epoch;
    unsigned long long timeout_ns;
    volatile int *abort_flag;    // in shared memory
};

constexpr uint32_t kTimeoutStatus = 6;  // SB_ERR_DEVICE_TIMEOUT

// Records `code` for launch `epoch` in the status word (epoch << 32) | code.  The word sits
// in caller memory that is never initialised, so it may hold anything: a word tagged with
// another epoch is replaced, and within the same epoch (CUDA-graph replays reuse theirs) the
// larger, i.e. worse, code is kept.
static __device__ __noinline__ void record_status(unsigned long long *status, uint32_t epoch,
                                                  uint32_t code) {
    const unsigned long long mine = (static_cast<unsigned long long>(epoch) << 32) | code;
    unsigned long long old = *reinterpret_cast<volatile unsigned long long *>(status);
    // each retry means another writer changed the word; a launch has only a few writers, so
    // the bound is never reached
    for (int tries = 0; tries < 4096; ++tries) {
        const bool same = static_cast<uint32_t>(old >> 32) == epoch;
        const unsigned long long want = (same && old > mine) ? old : mine;
        if (want == old) return;
        const unsigned long long seen = atomicCAS(status, old, want);
        if (seen == old) return;
        old = seen;
    }
}

// Scalars by value: a context passed by reference to an out-of-line function would be kept
// in local memory at every wait site.
static __device__ __noinline__ void raise_timeout(unsigned long long *status, uint32_t epoch,
                                                  volatile int *abort_flag) {
    *abort_flag = 1;
    record_status(status, epoch, kTimeoutStatus);
}

// Bounded wait on an mbarrier phase.  Returns false when the CTA is aborting (another role
// gave up) or when this wait itself runs out of time.
__device__ __forceinline__ bool bwait(uint64_t *bar, uint32_t parity, const WaitCtx w) {
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_test(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (*w.abort_flag) return false;
            if (globaltimer_ns() - t0 > w.timeout_ns) {
                raise_timeout(w.status, w.epoch, w.abort_flag);
                return false;
            }
        }
    }
}

// bwait for a barrier whose arrivals come from another CTA of the cluster (cluster-scope
// acquire).
__device__ __forceinline__ bool bwait_cluster(uint64_t *bar, uint32_t parity, const WaitCtx w) {
    if (mbar_test_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_test_cluster(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (*w.abort_flag) return false;
            if (globaltimer_ns() - t0 > w.timeout_ns) {
                raise_timeout(w.status, w.epoch, w.abort_flag);
                return false;
            }
        }
    }
}

// Bounded wait used while draining: ignores the abort flag (the copies or MMAs being waited
// for complete on their own), but still gives up after the time limit; false then.
__device__ __forceinline__ bool bwait_drain(uint64_t *bar, uint32_t parity, const WaitCtx w) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 0;; ++i) {
        if (mbar_test(bar, parity)) return true;
        if ((i & 63u) == 63u && globaltimer_ns() - t0 > w.timeout_ns) {
            raise_timeout(w.status, w.epoch, w.abort_flag);
            return false;
        }
    }
}

}  // namespace sb
