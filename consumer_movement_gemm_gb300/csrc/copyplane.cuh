// copyplane.cuh -- bulk row mover of the permuted copy (copy.cu).
//
// One warp streams its rows global -> shared -> global with bulk
// asynchronous copies through a ring of stages (the TMA 1-D row pipeline of
// the DeepEP FIFO-pipeline page: load a whole row into shared memory on an
// mbarrier, store it out as a bulk group).  Lane 0 issues every copy; the
// other lanes keep the pipeline's bookkeeping off that lane's critical path:
// they load the destination rows of the next 32 rows together (one load per
// lane, ahead of use) and, for a gated copy, count 32 retired rows at once --
// one acq_rel fence per lane, then 32 relaxed arrivals in flight together,
// the arrival that completes a chunk publishing its slot ("cross-GPU sync
// protocols on PCIe", section 3).  Store groups are retired LAG behind the
// newest; a row is counted only after its own store group has completed
// (writes done) and lane 0 has taken an async-proxy fence.
#pragma once
#include "ctrl.cuh"
#include "ptx.cuh"
#include "sync.cuh"

namespace tovl {

__device__ __forceinline__ void publish_chunk(const CopyParams& p, int c);

// Arrivals of this warp's rows [i0, i1) of batch `b` (rows 32b .. 32b + 31 of
// the warp's sequence; lane j holds the destination row of row 32b + j in
// `dst_of_lane`).  Every row's store has completed.
__device__ __forceinline__ void count_rows(const CopyParams& p, long long b, long long i0, long long i1, int dst_of_lane)
{
    const int lane = static_cast<int>(ptx::lane_id());
    const long long i = b * 32 + lane;
    __syncwarp();
    if (i >= i0 && i < i1) {
        ptx::fence_acq_rel_gpu();
        const int c = dst_of_lane / kChunkRows;
        const int old = ptx::atom_add_relaxed_gpu(p.ctrl.cnt + c * p.ctrl.n_slices, 1);
        if (old + 1 == p.seq * kChunkRows) publish_chunk(p, c);
    }
    __syncwarp();
}

// Stream rows first, first + step, ... (below p.n_rows) of the permuted copy.
// Row i of the sequence is held in stage i % ns.  Returns false on a
// pipeline timeout (after draining the loads in flight).
template <int LAG>
__device__ bool bulk_stream(const CopyParams& p, long long first, long long step, uint8_t* ring, uint64_t* bars, int ns,
                            uint32_t stride, long long timeout_ns)
{
    const int lane = static_cast<int>(ptx::lane_id());
    const uint32_t bytes = static_cast<uint32_t>(p.row_bytes);
    const long long n = first < p.n_rows ? (p.n_rows - first + step - 1) / step : 0;
    auto src_of = [&](long long i) { return p.src + (first + i * step) * p.row_bytes; };
    // destination row of sequence row 32b + lane (0 past the end)
    auto perm_batch = [&](long long b) {
        const long long i = b * 32 + lane;
        return i < n ? p.perm[first + i * step] : 0;
    };
    auto load = [&](long long i) {
        const int slot = static_cast<int>(i % ns);
        ptx::mbar_arrive_expect_tx(&bars[slot], bytes);
        ptx::bulk_load(ring + slot * stride, src_of(i), bytes, &bars[slot]);
    };
    int perm_prev = 0;
    int perm_cur = perm_batch(0);
    int perm_next = perm_batch(1);
    long long loaded = n < ns ? n : ns;
    if (lane == 0)
        for (long long i = 0; i < loaded; ++i) load(i);
    long long counted = 0;    // rows whose arrivals are done
    for (long long u = 0; u < n; ++u) {
        if (u > 0 && (u & 31) == 0) {
            perm_prev = perm_cur;
            perm_cur = perm_next;
            perm_next = perm_batch((u >> 5) + 1);
        }
        const int dst = __shfl_sync(0xffffffffu, perm_cur, static_cast<int>(u & 31));
        const int slot = static_cast<int>(u % ns);
        const bool ok = mbar_wait(&bars[slot], static_cast<uint32_t>((u / ns) & 1), p.ctrl, timeout_ns);
        if (!__all_sync(0xffffffffu, ok)) {
            // drain the loads still in flight before giving up
            if (lane == 0) {
                for (long long v = u + 1; v < loaded; ++v)
                    mbar_wait(&bars[v % ns], static_cast<uint32_t>((v / ns) & 1), p.ctrl, timeout_ns);
                ptx::bulk_wait<0>();
            }
            __syncwarp();
            return false;
        }
        if (lane == 0) {
            ptx::bulk_store(p.dst + static_cast<long long>(dst) * p.row_bytes, ring + slot * stride, bytes);
            ptx::bulk_commit();
        }
        if (u >= LAG) {
            // rows <= u - LAG are written; the stage of row u - LAG takes the next row
            if (lane == 0) ptx::bulk_wait<LAG>();
            if (loaded < n) {
                if (lane == 0) load(loaded);
                ++loaded;
            }
            const long long r = u - LAG;
            if (p.gated && (r & 31) == 31) {
                if (lane == 0) ptx::fence_proxy_async_global();
                count_rows(p, r >> 5, counted, r + 1, (r >> 5) == (u >> 5) ? perm_cur : perm_prev);
                counted = r + 1;
            }
        }
    }
    if (lane == 0) {
        ptx::bulk_wait<0>();
        ptx::fence_proxy_async_global();
    }
    __syncwarp();
    if (p.gated && n > 0) {
        // the last (at most two) partial batches
        const long long b_last = (n - 1) >> 5;
        if (counted < b_last * 32) count_rows(p, b_last - 1, counted, b_last * 32, perm_prev);
        count_rows(p, b_last, counted, n, perm_cur);
    }
    return true;
}

// Ring geometry inside `bytes_avail` bytes of shared memory: stage = one row
// rounded up to 128 B, at most kMaxRing stages; the mbarriers take the last
// 1 KB.
constexpr int kMaxRing = 32;

struct Ring {
    uint8_t* base;
    uint64_t* bars;
    int ns;
    uint32_t stride;
};

__device__ __forceinline__ Ring make_ring(uint8_t* smem, int bytes_avail, int row_bytes)
{
    Ring r;
    r.stride = (static_cast<uint32_t>(row_bytes) + 127u) & ~127u;
    const int usable = bytes_avail - 1024;
    int ns = usable / static_cast<int>(r.stride);
    r.ns = ns > kMaxRing ? kMaxRing : ns;
    r.base = smem;
    r.bars = reinterpret_cast<uint64_t*>(smem + usable);
    return r;
}

// Initialise the ring's barriers (lane 0) and run the stream with the
// deepest retire lag the ring allows.
__device__ inline bool run_bulk(const CopyParams& p, long long first, long long step, const Ring& r, long long timeout_ns)
{
    if (ptx::lane_id() == 0) {
        for (int i = 0; i < r.ns; ++i) ptx::mbar_init(&r.bars[i], 1);
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
    }
    __syncwarp();
    if (r.ns >= 16) return bulk_stream<8>(p, first, step, r.base, r.bars, r.ns, r.stride, timeout_ns);
    if (r.ns >= 8) return bulk_stream<4>(p, first, step, r.base, r.bars, r.ns, r.stride, timeout_ns);
    return bulk_stream<1>(p, first, step, r.base, r.bars, r.ns, r.stride, timeout_ns);
}

}  // namespace tovl
