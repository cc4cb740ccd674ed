// copyplane.cuh -- row movers for the data plane.
//
// bulk_stream: one issuing thread streams rows global -> shared -> global
// with bulk asynchronous copies through a ring of stages (the TMA 1-D row
// pipeline of the DeepEP FIFO-pipeline page: load a whole row into shared
// memory on an mbarrier, store it out as a bulk group).  Store groups are
// retired LAG behind the newest; a row is handed to job.done() only after its
// own store group has completed (writes visible), followed by an async-proxy
// fence, so the caller's release that follows covers the row.
#pragma once
#include "ctrl.cuh"
#include "ptx.cuh"
#include "sync.cuh"

namespace tovl {

// Job interface:
//   int next()                   next row id for this issuer, -1 when done
//   const void* src(int r)
//   void* dst(int r)
//   void done(int r)             the row's bytes are written and visible
template <int LAG, class Job>
__device__ bool bulk_stream(Job& job, uint32_t bytes, uint8_t* ring, uint64_t* bars, int* unit_row, int ns,
                            uint32_t stride, const Ctrl& ctrl, long long timeout_ns)
{
    auto load = [&](int slot, int r) {
        unit_row[slot] = r;
        ptx::mbar_arrive_expect_tx(&bars[slot], bytes);
        ptx::bulk_load(ring + slot * stride, job.src(r), bytes, &bars[slot]);
    };
    int loaded = 0;
    for (; loaded < ns; ++loaded) {
        const int r = job.next();
        if (r < 0) break;
        load(loaded, r);
    }
    for (int u = 0; u < loaded; ++u) {
        const int slot = u % ns;
        if (!mbar_wait(&bars[slot], (u / ns) & 1, ctrl, timeout_ns)) {
            // drain what is in flight before giving up
            for (int v = u + 1; v < loaded; ++v) mbar_wait(&bars[v % ns], (v / ns) & 1, ctrl, timeout_ns);
            ptx::bulk_wait<0>();
            return false;
        }
        ptx::bulk_store(job.dst(unit_row[slot]), ring + slot * stride, bytes);
        ptx::bulk_commit();
        if (u >= LAG) {
            ptx::bulk_wait<LAG>();
            ptx::fence_proxy_async_global();
            const int dslot = (u - LAG) % ns;
            job.done(unit_row[dslot]);
            const int nr = job.next();
            if (nr >= 0) {
                load(dslot, nr);
                ++loaded;
            }
        }
    }
    ptx::bulk_wait<0>();
    ptx::fence_proxy_async_global();
    for (int d = (loaded > LAG ? loaded - LAG : 0); d < loaded; ++d) job.done(unit_row[d % ns]);
    return true;
}

// Ring geometry inside `bytes_avail` bytes of shared memory: stage = one row
// rounded up to 128 B, at most kMaxRing stages; mbarriers and the unit table
// take the last 1 KB.
constexpr int kMaxRing = 32;

struct Ring {
    uint8_t* base;
    uint64_t* bars;
    int* unit_row;
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
    r.unit_row = reinterpret_cast<int*>(r.bars + kMaxRing);
    return r;
}

// Initialise the ring's barriers (one thread) and run the stream with the
// deepest retire lag the ring allows.
template <class Job>
__device__ bool run_bulk(Job& job, uint32_t bytes, const Ring& r, const Ctrl& ctrl, long long timeout_ns)
{
    for (int i = 0; i < r.ns; ++i) ptx::mbar_init(&r.bars[i], 1);
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
    if (r.ns >= 16) return bulk_stream<8>(job, bytes, r.base, r.bars, r.unit_row, r.ns, r.stride, ctrl, timeout_ns);
    if (r.ns >= 8) return bulk_stream<4>(job, bytes, r.base, r.bars, r.unit_row, r.ns, r.stride, ctrl, timeout_ns);
    return bulk_stream<1>(job, bytes, r.base, r.bars, r.unit_row, r.ns, r.stride, ctrl, timeout_ns);
}

}  // namespace tovl
