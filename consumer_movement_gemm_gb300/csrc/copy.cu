// copy.cu -- gated permuted row copy (the copy plane measured alone).
//
// dst[perm[i]] = src[i] for every source row i.  Chunks are 64 destination
// rows, so the 64 rows of a chunk come from many copier warps spread over the
// whole grid; each copied row is one arrival on its chunk counter and the
// arrival that completes the chunk publishes the round's sequence number into
// the chunk's slot ("cross-GPU sync protocols on PCIe", sections 3-4).
// Waiter CTAs poll every chunk slot with acquire loads, lane per slot, and
// stamp the first observation; the publisher stamps the publish time, so the
// signal-wait latency of every chunk is observe - publish.
// With gated == 0 the same copy loop runs with no counting at all (the
// ungated control); that call is not a protocol round.
#include <cuda_runtime.h>
#include "ctrl.cuh"
#include "ptx.cuh"
#include "sync.cuh"
#include "copyplane.cuh"
#include "launch.cuh"

namespace tovl {

constexpr int kCopyThreads = 512;
constexpr int kCopyUnroll = 8;
constexpr int kCopySmem = 200 * 1024;

// The elected arrival of chunk c (its relaxed add completed the count):
// acquire every earlier arrival, then publish the round's sequence.
__device__ __forceinline__ void publish_chunk(const CopyParams& p, int c)
{
    ptx::fence_acq_rel_gpu();
    if (p.stamps) p.ctrl.pub_ns[c] = static_cast<long long>(ptx::globaltimer());
    ptx::st_release_gpu(p.ctrl.slot + c * p.ctrl.n_slices, p.seq);
}

// Counters this copy does not fill to their per-round quota get the missing
// arrivals as one seed (partial last chunk, chunks beyond the copy, every
// row-block counter).
__device__ void copy_seeds(const CopyParams& p, int tid, int n_threads)
{
    const int S = p.ctrl.n_slices;
    for (int cs = tid; cs < p.ctrl.n_chunk_cap * S; cs += n_threads) {
        const int c = cs / S;
        const long long real = (cs % S) ? 0LL
                                        : min(max(p.n_rows - static_cast<long long>(c) * kChunkRows, 0LL),
                                              static_cast<long long>(kChunkRows));
        const int seed = kChunkRows - static_cast<int>(real);
        if (seed > 0) arrive_and_publish(p.ctrl, cs, seed, p.seq);
    }
    for (int bs = tid; bs < p.ctrl.n_block_cap * S; bs += n_threads)
        ptx::red_add_release_gpu(p.ctrl.rbcnt + bs, kBlockRows);
}

// Vector copy: each warp takes a group of consecutive source rows (about
// 16 KB) and moves it as one flat range of 16-byte words, kCopyUnroll words
// in flight per lane, the group's destination rows loaded once up front
// into a per-warp table in shared memory; then one lane per row counts the
// row.
__device__ void copy_v4(const CopyParams& p, int gw, int n_gw)
{
    __shared__ int dst_tabs[kCopyThreads / 32][64];
    const uint32_t lane = ptx::lane_id();
    int* dst_tab = dst_tabs[threadIdx.x / 32];
    const int n16 = p.row_bytes / 16;
    const int rows_per_group = min(64, max(1, 16384 / p.row_bytes));   // at most two rows per lane
    const long long n_groups = (p.n_rows + rows_per_group - 1) / rows_per_group;
    for (long long g = gw; g < n_groups; g += n_gw) {
        const long long r0 = g * rows_per_group;
        const int nr = static_cast<int>(min(static_cast<long long>(rows_per_group), p.n_rows - r0));
        const int total = nr * n16;
        // destination rows of the group's rows, loaded once (lane l those of
        // rows l and l + 32) into the warp's 64-entry table
        const int pd0 = static_cast<int>(lane) < nr ? p.perm[r0 + lane] : 0;
        const int pd1 = static_cast<int>(lane) + 32 < nr ? p.perm[r0 + lane + 32] : 0;
        __syncwarp();          // the previous group's stores have read the table
        dst_tab[lane] = pd0;
        dst_tab[lane + 32] = pd1;
        __syncwarp();
        for (int base = 0; base < total; base += 32 * kCopyUnroll) {
            int4 v[kCopyUnroll];
#pragma unroll
            for (int j = 0; j < kCopyUnroll; ++j) {
                const int idx = base + j * 32 + static_cast<int>(lane);
                if (idx < total) {
                    const int rr = idx / n16, cc = idx - rr * n16;
                    v[j] = ptx::ld_nc_v4(reinterpret_cast<const int4*>(p.src + (r0 + rr) * p.row_bytes) + cc);
                }
            }
#pragma unroll
            for (int j = 0; j < kCopyUnroll; ++j) {
                const int idx = base + j * 32 + static_cast<int>(lane);
                if (idx < total) {
                    const int rr = idx / n16, cc = idx - rr * n16;
                    const long long d = dst_tab[rr];
                    ptx::st_v4(reinterpret_cast<int4*>(p.dst + d * p.row_bytes) + cc, v[j]);
                }
            }
        }
        if (p.gated) {
            // One release fence covers the warp's row stores (ordered before
            // it by the warp barrier); the arrivals are then relaxed atomics,
            // so a lane's two arrivals are in flight together.  A lane whose
            // arrival completes a chunk takes an acquire fence before
            // publishing -- together the acq_rel counting of section 3.
            __syncwarp();
            ptx::fence_acq_rel_gpu();
            const int S = p.ctrl.n_slices;
            int c0 = -1, c1 = -1, o0 = 0, o1 = 0;
            if (static_cast<int>(lane) < nr) {
                c0 = pd0 / kChunkRows;
                o0 = ptx::atom_add_relaxed_gpu(p.ctrl.cnt + c0 * S, 1);
            }
            if (static_cast<int>(lane) + 32 < nr) {
                c1 = pd1 / kChunkRows;
                o1 = ptx::atom_add_relaxed_gpu(p.ctrl.cnt + c1 * S, 1);
            }
            if (c0 >= 0 && o0 + 1 == p.seq * kChunkRows) publish_chunk(p, c0);
            if (c1 >= 0 && o1 + 1 == p.seq * kChunkRows) publish_chunk(p, c1);
        }
    }
}

// Waiters: warp w watches chunks [w*per, (w+1)*per); lane i of the warp owns
// chunks c = base + i + 32*j.  A lane re-polls only chunks it has not seen.
// Eight slots per lane are read per pass with relaxed (strong) loads, so the
// eight reads are in flight together; a lane that sees a slot reach the
// round's sequence takes an acquire fence before it stamps the observation
// -- a strong read followed by the fence is an acquire of that slot (eight
// back-to-back acquire loads would each wait for the one before).
__device__ void copy_waiter(const CopyParams& p, int ww, int n_ww)
{
    const uint32_t lane = ptx::lane_id();
    const int per = (p.n_chunks + n_ww - 1) / n_ww;
    const int c0 = ww * per;
    const int c1 = min(p.n_chunks, c0 + per);
    if (c0 >= c1) return;
    const int cpl = (c1 - c0 + 31) / 32;          // chunks per lane
    const uint64_t start = ptx::globaltimer();
    int seen = 0, mine = 0;
    for (int j = 0; j < cpl; ++j)
        if (c0 + static_cast<int>(lane) + 32 * j < c1) ++mine;
    // seen bits for up to 64 chunks per lane; larger ranges fall back to a count
    unsigned long long seen_bits = 0ull;
    uint32_t backoff = 32;
    while (__any_sync(0xffffffffu, seen < mine)) {
        for (int j = 0; j < cpl && j < 64; j += 8) {
            int val[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int c = c0 + static_cast<int>(lane) + 32 * (j + u);
                val[u] = (j + u < cpl && c < c1 && !((seen_bits >> (j + u)) & 1ull)) ? ptx::ld_relaxed_gpu(p.ctrl.slot + c * p.ctrl.n_slices)
                                                                                        : -2147483647;
            }
            bool any = false;
#pragma unroll
            for (int u = 0; u < 8; ++u) any |= val[u] >= p.seq;
            if (any) ptx::fence_acq_rel_gpu();
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (val[u] >= p.seq) {
                    const int c = c0 + static_cast<int>(lane) + 32 * (j + u);
                    if (p.stamps) p.ctrl.obs_ns[c] = static_cast<long long>(ptx::globaltimer());
                    seen_bits |= 1ull << (j + u);
                    ++seen;
                }
            }
        }
        int stop = 0;
        if (lane == 0) {
            if (aborted(p.ctrl, p.seq)) {
                stop = 1;
            } else if (ptx::globaltimer() - start > static_cast<uint64_t>(p.timeout_ns)) {
                record_error(p.ctrl, kErrTimeout);
                raise_abort(p.ctrl, p.seq);
                stop = 1;
            }
        }
        if (__shfl_sync(0xffffffffu, stop, 0)) break;
        __nanosleep(backoff);
        if (backoff < 128) backoff <<= 1;
    }
}

__global__ void __launch_bounds__(kCopyThreads, 2) copy_kernel(const __grid_constant__ CopyParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const int warp = threadIdx.x / 32;
    const int n_warps = kCopyThreads / 32;
    if (static_cast<int>(blockIdx.x) >= p.n_copiers) {
        copy_waiter(p, (blockIdx.x - p.n_copiers) * n_warps + warp, (gridDim.x - p.n_copiers) * n_warps);
        return;
    }
    if (p.gated) copy_seeds(p, blockIdx.x * kCopyThreads + threadIdx.x, p.n_copiers * kCopyThreads);
    if (p.copy_mode == 0) {
        copy_v4(p, blockIdx.x * n_warps + warp, p.n_copiers * n_warps);
        return;
    }
    // bulk mode: four warps each stream rows through a quarter of the shared
    // memory (lane 0 issues the copies; the warp prefetches destinations and
    // counts retired rows 32 at a time)
    constexpr int kIssuers = 4;
    if (warp < kIssuers) {
        uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
        const int share = (kCopySmem - 1024) / kIssuers / 1024 * 1024;
        const Ring ring = make_ring(smem + warp * share, share, p.row_bytes);
        run_bulk(p, static_cast<long long>(blockIdx.x) * kIssuers + warp, static_cast<long long>(p.n_copiers) * kIssuers,
                 ring, p.pipe_timeout_ns);
    }
}

}  // namespace tovl

namespace tovl {

// Waiter CTAs spin on slots the copier CTAs publish, so a gated copy asks
// for the cooperative co-residency guarantee (unless `cooperative` is off, for
// tools that cannot replay cooperative launches; the grid is sized to fit the
// device either way).
cudaError_t launch_copy(const CopyParams& p, int n_waiters, bool cooperative, cudaStream_t stream)
{
    const int grid = p.n_copiers + n_waiters;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(grid);
    lc.blockDim = dim3(kCopyThreads);
    lc.dynamicSmemBytes = p.copy_mode ? kCopySmem : 0;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = (cooperative && n_waiters > 0) ? 1 : 0;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, copy_kernel, p);
}

cudaError_t prepare_copy()
{
    return cudaFuncSetAttribute(copy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kCopySmem);
}

int copy_max_active_per_sm(int copy_mode)
{
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, copy_kernel, kCopyThreads, copy_mode ? kCopySmem : 0) !=
        cudaSuccess)
        return 0;
    return n;
}

int copy_bulk_max_row_bytes()
{
    // each of the four issuers needs at least two stages in its share
    return ((kCopySmem - 1024) / 4 / 1024 * 1024 - 1024) / 2 / 128 * 128;
}

}  // namespace tovl
