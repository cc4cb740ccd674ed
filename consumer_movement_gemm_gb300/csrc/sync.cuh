// sync.cuh -- the single-writer completion protocol on one GPU.
//
// "Cross-GPU sync protocols on PCIe" (Astro Bear, part 4):
//   section 2  a slot has exactly one writer, which release-stores a
//              monotonically increasing sequence number; a waiter polls its
//              local slot with acquire loads until the value is >= seq.
//   section 3  a completion made of many writers is counted with a local
//              acq_rel atomic; the arrival that brings the count to its target
//              is elected and becomes the slot's single writer.
//   section 4  one slot per 64-row chunk (watermark), not per row or tile.
//   section 5  local row-block counters take release reductions; rows that
//              nobody writes (padding) are pre-seeded into the counter.
// Every wait here is bounded (DeepEP pipeline page: timeout_while); on expiry
// the waiter records TIMEOUT in the sticky status word, raises the launch's
// abort sequence so the other waiters stop, and returns without trapping.
#pragma once
#include "ctrl.cuh"
#include "ptx.cuh"

namespace tovl {

__device__ __forceinline__ void record_error(const Ctrl& c, int code)
{
    ptx::atom_cas_relaxed_gpu(c.status, kOk, code);
}

__device__ __forceinline__ void raise_abort(const Ctrl& c, int seq)
{
    ptx::atom_max_relaxed_gpu(c.abort_seq, seq);
}

__device__ __forceinline__ bool aborted(const Ctrl& c, int seq)
{
    return ptx::ld_relaxed_gpu(c.abort_seq) >= seq;
}

// Count `n` arrivals on chunk `c` for round `seq`.  The arrival that brings
// the monotonic counter to seq * kChunkRows publishes `seq` into the chunk's
// slot with a release store.  Returns true for the elected publisher.
__device__ __forceinline__ bool arrive_and_publish(const Ctrl& ctrl, int c, int n, int seq)
{
    const int old = ptx::atom_add_acq_rel_gpu(ctrl.cnt + c, n);
    if (old + n == seq * kChunkRows) {
        ptx::st_release_gpu(ctrl.slot + c, seq);
        return true;
    }
    return false;
}

// Bounded wait of one warp until every watched word is >= target.
// Lane i watches words[i] (lanes >= n watch nothing).  Polls use acquire
// loads; the warp decides with a vote.  The lane that saw a word reach the
// target holds an acquire observation of it; the warp barrier after the vote
// orders every lane's observation before whatever any lane of the warp does
// next (bar.warp.sync orders memory among its threads), so lane 0 may hand
// the gate on without reading the words again.  Returns the number of
// polling rounds, negative on timeout or abort.
__device__ __forceinline__ int warp_wait_lanes(const int* mine, int target, const Ctrl& ctrl, int seq,
                                               long long timeout_ns);

__device__ __forceinline__ int warp_wait_ge(const int* const* words, int n, int target, const Ctrl& ctrl, int seq,
                                            long long timeout_ns)
{
    const uint32_t lane = ptx::lane_id();
    return warp_wait_lanes((static_cast<int>(lane) < n) ? words[lane] : nullptr, target, ctrl, seq, timeout_ns);
}

// The same wait with each lane naming its own word (nullptr: none).
__device__ __forceinline__ int warp_wait_lanes(const int* mine, int target, const Ctrl& ctrl, int seq,
                                               long long timeout_ns)
{
    const uint32_t lane = ptx::lane_id();
    uint64_t start = 0;
    int rounds = 0;
    uint32_t backoff = 32;
    for (;;) {
        ++rounds;
        const bool ok = (mine == nullptr) || (ptx::ld_acquire_gpu(mine) >= target);
        if (__all_sync(0xffffffffu, ok)) break;
        if ((rounds & 15) == 1) {
            int stop = 0;
            if (lane == 0) {
                const uint64_t now = ptx::globaltimer();
                if (start == 0) start = now;
                if (aborted(ctrl, seq)) stop = 1;
                else if (now - start > static_cast<uint64_t>(timeout_ns)) {
                    record_error(ctrl, kErrTimeout);
                    raise_abort(ctrl, seq);
                    stop = 2;
                }
            }
            stop = __shfl_sync(0xffffffffu, stop, 0);
            if (stop) return -rounds;
        }
        __nanosleep(backoff);
        if (backoff < 256) backoff <<= 1;
    }
    __syncwarp();
    return rounds;
}

// Bounded mbarrier wait (intra-CTA pipelines).  These only depend on this
// CTA's own asynchronous copies and MMAs; the bound guards against a logic
// error turning into a hung GPU.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const Ctrl& ctrl, long long timeout_ns)
{
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t start = ptx::globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((i & 255) == 0 && ptx::globaltimer() - start > static_cast<uint64_t>(timeout_ns)) {
            record_error(ctrl, kErrTimeout);
            return false;
        }
    }
}

}  // namespace tovl
