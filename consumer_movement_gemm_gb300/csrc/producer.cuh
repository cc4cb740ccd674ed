// producer.cuh -- producer CTAs of the fused kernel: row copies and arrivals.
//
// Producers copy token rows into the gathered (or dispatched) buffer with
// 16-byte vector loads/stores and count them with the single-writer protocol
// ("cross-GPU sync protocols on PCIe", sections 3-5): an acq_rel arrival per
// item on its chunk-slice counter, the arrival that completes the count
// release-stores the round's sequence into the slot (gather), or release
// reductions into row-block counters pre-seeded with the padding (dispatch).
// Items follow the consumers' traversal order (section 6, item 3).
#pragma once
#include "ctrl.cuh"
#include "ptx.cuh"
#include "sync.cuh"
#include "common.cuh"

namespace tovl {

// Row-block-slice items: item i -> (row block mb, K-slice s, row group q)
// in the consumers' order: groups of wave_blocks row blocks, each group slice
// by slice, each slice block by block.
struct Item {
    int mb, s, r0;
};

__device__ __forceinline__ Item decode_item(const FusedParams& p, int i, int n_blocks)
{
    const int ipb = kBlockRows / p.item_rows;              // items per block per slice
    const int per_group = p.wave_blocks * p.k_slices * ipb;
    const int g = i / per_group;
    const int b0 = g * p.wave_blocks;
    const int gs = min(p.wave_blocks, n_blocks - b0);
    const int rem = i - g * per_group;
    Item it;
    it.s = rem / (gs * ipb);
    const int rem2 = rem - it.s * gs * ipb;
    it.mb = b0 + rem2 / ipb;
    it.r0 = it.mb * kBlockRows + (rem2 % ipb) * p.item_rows;
    return it;
}

// Source address of destination row r (nullptr: no source, padding row).
__device__ __forceinline__ const uint8_t* row_src(const FusedParams& p, int r)
{
    if (p.mode == kModeGather) {
        if (r >= p.M) return nullptr;
        const int s = r / p.rows_per_shard;
        const int i = r - s * p.rows_per_shard;
        return static_cast<const uint8_t*>(p.shard[s]) + static_cast<size_t>(i) * p.row_bytes;
    }
    const int t = p.src_of_dst[r];
    return t < 0 ? nullptr : static_cast<const uint8_t*>(p.x) + static_cast<size_t>(t) * p.row_bytes;
}

// Counter index and completion of an item's rows.
__device__ __forceinline__ void item_done(const FusedParams& p, int counter, int n)
{
    if (p.mode == kModeGather) {
        if (arrive_and_publish(p.ctrl, counter, n, p.seq) && p.stats)
            p.ctrl.pub_ns[counter] = static_cast<long long>(ptx::globaltimer());
    } else {
        ptx::red_add_release_gpu(p.ctrl.rbcnt + counter, n);
    }
}

// Per-round padding seeds.  Each counter must gain exactly its per-round
// quota (64 per chunk slice, 128 per block slice) every call, so whatever
// this call does not fill -- rows past the end, padding rows, slices beyond
// k_slices, blocks beyond this round -- is added as one seed.
// Seeds come in two phases.  Completion seeds -- the padding of a partial
// chunk or of a dispatch row block -- are part of a gate's target, so they
// are added before any row is copied.  Quota seeds -- counters this call
// does not use at all (chunks past the rows, slices past k_slices, the other
// counter family) -- only keep the closed form, so they are added after the
// copies, off the consumers' critical path.
__device__ void seed_counters(const FusedParams& p, int gw, int n_gw, bool completion)
{
    const uint32_t lane = ptx::lane_id();
    const Ctrl& c = p.ctrl;
    const int S = c.n_slices;
    // chunk-slice counters
    for (int cs = gw * 32 + lane; cs < c.n_chunk_cap * S; cs += n_gw * 32) {
        const int ch = cs / S, sl = cs - ch * S;
        int real = 0;
        if (p.mode == kModeGather && sl < p.k_slices) real = min(max(p.M - ch * kChunkRows, 0), kChunkRows);
        const bool is_completion = real > 0 && real < kChunkRows;
        if (is_completion == completion && real < kChunkRows) arrive_and_publish(c, cs, kChunkRows - real, p.seq);
    }
    // block-slice counters
    if (p.mode == kModeGather) {
        if (!completion)
            for (int bs = gw * 32 + lane; bs < c.n_block_cap * S; bs += n_gw * 32)
                ptx::red_add_release_gpu(c.rbcnt + bs, kBlockRows);
        return;
    }
    const int n_blocks = p.meta[1];
    const int zero = p.meta[2];
    for (int b = gw; b < c.n_block_cap; b += n_gw) {
        if (b >= n_blocks) {
            if (!completion && static_cast<int>(lane) < S) ptx::red_add_release_gpu(c.rbcnt + b * S + lane, kBlockRows);
            continue;
        }
        const int pad = p.pad[b];
        if (completion && zero && pad > 0) {
            // padding rows are the last `pad` rows of the block; they must be
            // zero before the counters reach their target
            int4* d = reinterpret_cast<int4*>(static_cast<uint8_t*>(p.gathered) +
                                              static_cast<size_t>(b * kBlockRows + kBlockRows - pad) * p.row_bytes);
            const size_t n16 = static_cast<size_t>(pad) * p.row_bytes / 16;
            const int4 z = make_int4(0, 0, 0, 0);
            for (size_t i = lane; i < n16; i += 32) ptx::st_v4(d + i, z);
            __syncwarp();
        }
        // slices in use get the padding count (completion), slices beyond
        // k_slices the whole block quota (quota)
        if (static_cast<int>(lane) < S) {
            const bool used = static_cast<int>(lane) < p.k_slices;
            const int seed = used ? pad : kBlockRows;
            if (used == completion && seed > 0) ptx::red_add_release_gpu(c.rbcnt + b * S + lane, seed);
        }
    }
}

// Copy one item: item_rows destination rows x the K-slice's bytes, as one
// flat range of 16-byte words walked 32 words per step, 16 words per lane in
// flight.  A per-warp table in shared memory holds each row's source.
__device__ __forceinline__ int copy_item(const FusedParams& p, const Item& it, const uint8_t** tbl)
{
    const uint32_t lane = ptx::lane_id();
    const int RI = p.item_rows;
    for (int l = lane; l < RI; l += 32) tbl[l] = row_src(p, it.r0 + l);
    __syncwarp();
    const size_t soff = static_cast<size_t>(kb_begin(p, it.s)) * kTileK * 2;
    const int n16 = (kb_begin(p, it.s + 1) - kb_begin(p, it.s)) * kTileK * 2 / 16;
    uint8_t* dst = static_cast<uint8_t*>(p.gathered) + soff + static_cast<size_t>(it.r0) * p.row_bytes;
    // lane position (row, col) in the item's flat range, advanced by 32 words
    // per step without division
    int row = static_cast<int>(lane) / n16;
    int col = static_cast<int>(lane) - row * n16;
    while (row < RI) {
        int4 v[kItemInt4 / 32];
        int r = row, c = col;
#pragma unroll
        for (int j = 0; j < kItemInt4 / 32; ++j) {
            if (r < RI) {
                const uint8_t* src = tbl[r];
                if (src) v[j] = ptx::ld_nc_v4(reinterpret_cast<const int4*>(src + soff) + c);
            }
            c += 32;
            while (c >= n16) {
                c -= n16;
                ++r;
            }
        }
        r = row;
        c = col;
#pragma unroll
        for (int j = 0; j < kItemInt4 / 32; ++j) {
            if (r < RI && tbl[r]) ptx::st_v4(reinterpret_cast<int4*>(dst + static_cast<size_t>(r) * p.row_bytes) + c, v[j]);
            c += 32;
            while (c >= n16) {
                c -= n16;
                ++r;
            }
        }
        row = r;
        col = c;
    }
    // rows this item filled
    int n = 0;
    for (int l = 0; l < RI; l += 32) {
        const bool real = (l + static_cast<int>(lane) < RI) && tbl[l + lane] != nullptr;
        n += __popc(__ballot_sync(0xffffffffu, real));
    }
    __syncwarp();
    return n;
}

__device__ void producer(const FusedParams& p, uint8_t* smem, int pid)
{
    const int warp = threadIdx.x / 32;
    const uint32_t lane = ptx::lane_id();
    const int n_warps = kThreads / 32;
    // consecutive items go to different CTAs (SMs), so the rows of one chunk
    // are copied by many SMs at once
    const int gw = warp * p.n_producers + pid;
    const int n_gw = p.n_producers * n_warps;
    if (threadIdx.x == 0) stat_min(p, kStatProdStartNs, ptx::globaltimer());
    seed_counters(p, gw, n_gw, true);

    const uint8_t** tbl = reinterpret_cast<const uint8_t**>(smem) + warp * 64;   // row-source table per warp
    const int n_blocks = num_row_blocks(p);
    const int n_items = n_blocks * p.k_slices * (kBlockRows / p.item_rows);
    const int S = p.ctrl.n_slices;
    // Every item is released as soon as it is copied: a warp's consecutive
    // items are n_gw items apart in the consumers' order, so holding one back
    // to share a release fence would delay an earlier K-slice behind later
    // ones (measured: batching four items cost 12 us of the TP fused call and
    // saved no copy time).
    for (int i = gw; i < n_items; i += n_gw) {
        const Item it = decode_item(p, i, n_blocks);
        const int n = copy_item(p, it, tbl);
        const int counter = (p.mode == kModeGather) ? (it.r0 / kChunkRows) * S + it.s : it.mb * S + it.s;
        // the copies above happen-before lane 0's release below
        __syncwarp();
        if (lane == 0 && n > 0) item_done(p, counter, n);
        __syncwarp();
    }
    seed_counters(p, gw, n_gw, false);
    __syncwarp();
    __syncthreads();
    if (threadIdx.x == 0) stat_max(p, kStatProdEndNs, ptx::globaltimer());
}

}  // namespace tovl
