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
        if (r >= gather_rows(p)) return nullptr;
        if (p.src_rows) return static_cast<const uint8_t*>(p.x) + static_cast<size_t>(p.src_rows[r]) * p.row_bytes;
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
__device__ inline void seed_counters(const FusedParams& p, int gw, int n_gw, bool completion)
{
    const uint32_t lane = ptx::lane_id();
    const Ctrl& c = p.ctrl;
    const int S = c.n_slices;
    // chunk-slice counters
    for (int cs = gw * 32 + lane; cs < c.n_chunk_cap * S; cs += n_gw * 32) {
        const int ch = cs / S, sl = cs - ch * S;
        int real = 0;
        if (p.mode == kModeGather && sl < p.k_slices) real = min(max(gather_rows(p) - ch * kChunkRows, 0), kChunkRows);
        // reduce-scatter: counter t collects the quota from partial tile t's epilogue warps
        if (p.mode == kModeReduceScatter && cs < p.rs_tiles) real = kChunkRows;
        const bool is_completion = real > 0 && real < kChunkRows;
        if (is_completion == completion && real < kChunkRows) arrive_and_publish(c, cs, kChunkRows - real, p.seq);
    }
    // block-slice counters
    if (p.mode == kModeGather || p.mode == kModeReduceScatter) {
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

// Lane layout of one item.  An item is RI rows x n16 16-byte words; G rows
// are copied at once, L = 32 / G lanes per row, each lane owning M = RI / G
// rows (M > 1 only when RI > 16).  Lane l copies words lo, lo + L, lo + 2L,
// ... of rows lr + G*m (lr = l / L, lo = l % L): every group of L lanes moves
// L x 16 contiguous bytes (at least one full 32-byte sector) per instruction,
// each lane keeps one source and one destination pointer per row, and the
// word offsets of a pass are compile-time multiples of L x 16 bytes.
template <int M>
struct ItemState {
    Item it;
    const uint8_t* src[M];   // this lane's rows (a readable dummy where a row has no source)
    uint8_t* dst[M];
    bool has[M];             // the row has a source
    int n16;                 // 16-byte words per row slice
    int counter;
    int n;                   // rows of this item that have a source
};

template <int M>
struct LaneMap {
    int RI, G, L, lr, lo;
    __device__ LaneMap(int ri, int lane)
    {
        RI = ri;
        G = ri / M;
        L = 32 / G;
        lr = lane / L;
        lo = lane - lr * L;
    }
};

// Decode item i and resolve this lane's rows.
template <int M>
__device__ __forceinline__ ItemState<M> begin_item(const FusedParams& p, const LaneMap<M>& lm, int i, int n_blocks)
{
    const int lane = static_cast<int>(ptx::lane_id());
    // a readable row for lanes whose row has no source: the shards' first
    // row for an all-gather, the source buffer for a row table or a dispatch
    const uint8_t* dummy =
        static_cast<const uint8_t*>((p.mode == kModeGather && !p.src_rows) ? p.shard[0] : p.x);
    ItemState<M> st;
    st.it = decode_item(p, i, n_blocks);
    const size_t soff = static_cast<size_t>(kb_begin(p, st.it.s)) * kTileK * 2;
    st.n16 = (kb_begin(p, st.it.s + 1) - kb_begin(p, st.it.s)) * kTileK * 2 / 16;
    st.counter = (p.mode == kModeGather) ? (st.it.r0 / kChunkRows) * p.ctrl.n_slices + st.it.s
                                         : st.it.mb * p.ctrl.n_slices + st.it.s;
    // lanes l < RI resolve rows l and l + 32; the row owners read them by shuffle
    const uint8_t* s0 = lane < lm.RI ? row_src(p, st.it.r0 + lane) : nullptr;
    const uint8_t* s1 = lane + 32 < lm.RI ? row_src(p, st.it.r0 + lane + 32) : nullptr;
    st.n = __popc(__ballot_sync(0xffffffffu, s0 != nullptr)) + __popc(__ballot_sync(0xffffffffu, s1 != nullptr));
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const int r = lm.lr + lm.G * m;
        const unsigned long long a0 = __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(s0), r & 31);
        const unsigned long long a1 = __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(s1), r & 31);
        const uint8_t* src = reinterpret_cast<const uint8_t*>(r < 32 ? a0 : a1);
        st.has[m] = src != nullptr;
        st.src[m] = src ? src + soff : dummy;
        st.dst[m] = static_cast<uint8_t*>(p.gathered) + static_cast<size_t>(st.it.r0 + r) * p.row_bytes + soff;
    }
    return st;
}

// Pass `ps` over an item: 16 words per lane.  Loads are unconditional (a
// word outside the item reads the row's first word, or the dummy row): a
// conditional load into a live register must be merged with the old value,
// which makes every load wait for the one before it.
template <int M>
__device__ __forceinline__ void load_pass(const ItemState<M>& st, const LaneMap<M>& lm, int ps,
                                          int4 (&v)[kItemInt4 / 32], uint64_t pol)
{
    constexpr int QN = kItemInt4 / 32 / M;    // words per row per lane and pass
#pragma unroll
    for (int k = 0; k < kItemInt4 / 32; ++k) {
        const int m = k / QN, q = k % QN;
        const int c = lm.lo + lm.L * (ps * QN + q);
        const int4* a = reinterpret_cast<const int4*>(st.src[m]) + (c < st.n16 ? c : 0);
        v[k] = ptx::ld_nc_v4_hint(a, pol);
    }
}

template <int M>
__device__ __forceinline__ void store_pass(const ItemState<M>& st, const LaneMap<M>& lm, int ps,
                                           const int4 (&v)[kItemInt4 / 32], uint64_t pol)
{
    constexpr int QN = kItemInt4 / 32 / M;
#pragma unroll
    for (int k = 0; k < kItemInt4 / 32; ++k) {
        const int m = k / QN, q = k % QN;
        const int c = lm.lo + lm.L * (ps * QN + q);
        if (st.has[m] && c < st.n16) ptx::st_v4_hint(reinterpret_cast<int4*>(st.dst[m]) + c, v[k], pol);
    }
}

template <int M>
__device__ void copy_items(const FusedParams& p, int gw, int n_gw)
{
    const int lane = static_cast<int>(ptx::lane_id());
    const LaneMap<M> lm(p.item_rows, lane);
    const int n_blocks = num_row_blocks(p);
    const int n_items = n_blocks * p.k_slices * (kBlockRows / p.item_rows);
    // words a lane covers per pass, per row: QN words L apart
    const int per_pass = lm.L * (kItemInt4 / 32 / M);
    const uint64_t pol_src = stream_policy(p, kHintSrcLast, kHintSrcFirst);
    const uint64_t pol_dst = stream_policy(p, kHintDstLast, 0);
    // Every item is released as soon as it is copied: a warp's consecutive
    // items are n_gw items apart in the consumers' order, so holding one back
    // to share a release fence would delay an earlier K-slice behind later
    // ones (measured: batching four items cost 12 us of the TP fused call and
    // saved no copy time).  Issuing the next item's loads before this item's
    // release was measured too: the release then also waits for those loads,
    // and the first chunks publish later.
    for (int i = gw; i < n_items; i += n_gw) {
        const ItemState<M> st = begin_item<M>(p, lm, i, n_blocks);
        const int passes = (st.n16 + per_pass - 1) / per_pass;
        for (int ps = 0; ps < passes; ++ps) {
            int4 v[kItemInt4 / 32];
            load_pass<M>(st, lm, ps, v, pol_src);
            store_pass<M>(st, lm, ps, v, pol_dst);
        }
        // the copies above happen-before lane 0's release below
        __syncwarp();
        if (lane == 0 && st.n > 0) item_done(p, st.counter, st.n);
        __syncwarp();
    }
}

// Staged variant: each warp owns an 8 KB shared-memory buffer and an
// mbarrier.  Per pass, the lanes that own rows issue bulk asynchronous loads
// of their row segments into the buffer (completion counted in bytes on the
// warp's mbarrier); the warp waits, then writes the buffer out with 16-byte
// vector stores in the lane layout above.  The loads in flight live in the
// producer CTA's shared memory, which it has no other use for, instead of
// in L1.
template <int M>
__device__ void copy_items_staged(const FusedParams& p, uint8_t* smem, int gw, int n_gw)
{
    const int lane = static_cast<int>(ptx::lane_id());
    const int warp = threadIdx.x / 32;
    uint8_t* buf = smem + warp * kItemBytes;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + (kThreads / 32) * kItemBytes) + warp;
    if (lane == 0) {
        ptx::mbar_init(bar, 1);
        ptx::fence_mbar_init();
    }
    __syncwarp();
    uint32_t phase = 0;
    const LaneMap<M> lm(p.item_rows, lane);
    const int RI = p.item_rows;
    const int n_blocks = num_row_blocks(p);
    const int n_items = n_blocks * p.k_slices * (kBlockRows / RI);
    constexpr int QN = kItemInt4 / 32 / M;
    for (int i = gw; i < n_items; i += n_gw) {
        const ItemState<M> st = begin_item<M>(p, lm, i, n_blocks);
        const size_t soff = static_cast<size_t>(kb_begin(p, st.it.s)) * kTileK * 2;
        const int passes = (st.n16 + kItemInt4 - 1) / kItemInt4;   // > 1 only for single-row items
        for (int ps = 0; ps < passes && st.n > 0; ++ps) {
            const int words = min(st.n16 - ps * kItemInt4, kItemInt4 / RI);   // 16-byte words per row this pass
            const uint32_t seg = static_cast<uint32_t>(words) * 16;
            if (lane == 0) ptx::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(st.n) * seg);
            __syncwarp();
            for (int l = lane; l < RI; l += 32) {
                const uint8_t* src = row_src(p, st.it.r0 + l);
                if (src) ptx::bulk_load(buf + l * seg, src + soff + static_cast<size_t>(ps) * kItemBytes, seg, bar);
            }
            const bool ok = mbar_wait(bar, phase, p.ctrl, p.pipe_timeout_ns);
            phase ^= 1u;
            if (!__all_sync(0xffffffffu, ok)) return;
            const uint32_t base = ptx::smem_u32(buf);
#pragma unroll
            for (int k = 0; k < kItemInt4 / 32; ++k) {
                const int m = k / QN, q = k % QN;
                const int r = lm.lr + lm.G * m;
                const int c = lm.lo + lm.L * q;
                if (st.has[m] && c < words) {
                    const int4 v = ptx::ld_shared_v4(base + static_cast<uint32_t>(r) * seg + c * 16);
                    ptx::st_v4(reinterpret_cast<int4*>(st.dst[m]) + ps * kItemInt4 + c, v);
                }
            }
            // the buffer's generic reads come before the next pass's bulk writes
            ptx::fence_proxy_async_smem();
            __syncwarp();
        }
        // the copies above happen-before lane 0's release below
        __syncwarp();
        if (lane == 0 && st.n > 0) item_done(p, st.counter, st.n);
        __syncwarp();
    }
    // every load this warp issued has completed; the barrier's memory may be
    // reused (a producer CTA that turns consumer)
    if (lane == 0) ptx::mbar_inval(bar);
    __syncwarp();
}

// Reduce-scatter reduction.  An item is 16 rows x 256 columns of one output
// tile; items are numbered in the consumers' tile order and handed out by a
// per-round ticket counter, so any warp that is free -- a producer warp from
// the start, a consumer warp once its CTA's tiles are done (the role switch)
// -- takes the next one.  For each item the warp waits until the S partial
// tiles of its output tile are published (lane s polls tile s's slot with
// acquire loads; warp vote; 32 shards per pass), then sums the S bf16 partials of its rows in
// fp32, ascending s, and stores the bf16 result, four rows at a time.  Lane l
// owns the 16-byte column group l of each row (32 groups = 256 columns).
// Shards are read four at a time, so each lane has 16 loads in flight.
static __device__ __noinline__ void rs_reduce(const FusedParams& p)
{
    constexpr int kItemRows = 16;
    constexpr int kRows = 4;
    constexpr int kShardsAtOnce = 4;
    const int lane = static_cast<int>(ptx::lane_id());
    const int S = p.n_shards;
    const int M = p.M;
    const int tile_rows = kTileM * p.rs_pair;
    const int per_tile = tile_rows / kItemRows;
    const int n_out = p.rs_tiles / S;
    const int n_items = n_out * per_tile;
    const size_t row_bytes = static_cast<size_t>(p.N) * 2;
    const size_t shard_bytes = static_cast<size_t>(M) * row_bytes;
    const uint8_t* part = static_cast<const uint8_t*>(p.out);
    uint8_t* out = static_cast<uint8_t*>(p.rs_out);
    for (;;) {
        int i = 0;
        if (lane == 0) i = ptx::atom_add_relaxed_gpu(p.ctrl.work, 1);
        i = __shfl_sync(0xffffffffu, i, 0);
        if (i >= n_items) break;
        const int u = i / per_tile;
        const int item_r0 = (u / p.n_nb) * tile_rows + (i - u * per_tile) * kItemRows;
        if (item_r0 >= M) continue;
        bool ok = true;
        for (int s0 = 0; s0 < S && ok; s0 += 32)     // lane s polls shard s0 + s (up to 64 shards)
            ok = warp_wait_lanes(s0 + lane < S ? p.ctrl.slot + u * S + s0 + lane : nullptr, p.gate_seq, p.ctrl, p.seq,
                                 p.timeout_ns) >= 0;
        if (!ok) return;
        const size_t col = static_cast<size_t>(u % p.n_nb) * kTileN * 2 + static_cast<size_t>(lane) * 16;
#pragma unroll 1
        for (int r0 = item_r0; r0 < item_r0 + kItemRows; r0 += kRows) {
            const uint8_t* base = part + static_cast<size_t>(r0) * row_bytes + col;
            float acc[kRows][8];
#pragma unroll
            for (int j = 0; j < kRows; ++j)
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[j][c] = 0.0f;
            for (int s0 = 0; s0 < S; s0 += kShardsAtOnce) {
                int4 v[kShardsAtOnce][kRows];
#pragma unroll
                for (int q = 0; q < kShardsAtOnce; ++q) {
                    // shards past S re-read the last one (unconditional loads; their sums are skipped)
                    const int s = min(s0 + q, S - 1);
#pragma unroll
                    for (int j = 0; j < kRows; ++j)
                        v[q][j] = ptx::ld_v4(reinterpret_cast<const int4*>(base + s * shard_bytes + j * row_bytes));
                }
#pragma unroll
                for (int q = 0; q < kShardsAtOnce; ++q) {
                    if (s0 + q >= S) break;
#pragma unroll
                    for (int j = 0; j < kRows; ++j) {
                        const uint32_t w[4] = {static_cast<uint32_t>(v[q][j].x), static_cast<uint32_t>(v[q][j].y),
                                               static_cast<uint32_t>(v[q][j].z), static_cast<uint32_t>(v[q][j].w)};
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            acc[j][2 * c] = __fadd_rn(acc[j][2 * c], __uint_as_float(w[c] << 16));
                            acc[j][2 * c + 1] = __fadd_rn(acc[j][2 * c + 1], __uint_as_float(w[c] & 0xffff0000u));
                        }
                    }
                }
            }
            uint8_t* dst = out + static_cast<size_t>(r0) * row_bytes + col;
#pragma unroll
            for (int j = 0; j < kRows; ++j) {
                int4 o;
                o.x = static_cast<int>(ptx::pack_bf16x2(acc[j][0], acc[j][1]));
                o.y = static_cast<int>(ptx::pack_bf16x2(acc[j][2], acc[j][3]));
                o.z = static_cast<int>(ptx::pack_bf16x2(acc[j][4], acc[j][5]));
                o.w = static_cast<int>(ptx::pack_bf16x2(acc[j][6], acc[j][7]));
                ptx::st_v4(reinterpret_cast<int4*>(dst + j * row_bytes), o);
            }
        }
    }
}

// Reduce-scatter reduction by the partial tiles' own CTAs (rs_epi).  The CTA
// (pair) that computes shard (o mod S)'s partial of output tile o also sums
// that tile, in `n_warps` warps that are otherwise idle in this launch
// (warps first_warp..15): for each of this CTA's tiles it owns, they wait
// until all S partials of the tile are published (lane s polls partial tile
// o*S + s's slot with acquire loads, warp vote, 32 shards per pass), then
// reduce this CTA's 128 rows x 256 columns of it,
//   out[m][n] = bf16( sum_s f32(P_s[m][n]) ), fp32 sums in ascending s,
// reading the partials from global memory, where they were stored
// microseconds earlier (L2).  A warp takes rows w, w + n_warps, ...; one row
// of the tile is 32 lanes x 16 bytes, and four rows of four shards are loaded
// together (16 loads in flight per lane).  The epilogue warps never wait on
// these warps, so a reduction overlaps the following tiles.
constexpr int kRsRows = 4;        // rows per batch
constexpr int kRsShards = 4;      // shards loaded together

static __device__ __noinline__ void rs_reduce_owned(const FusedParams& p, int unit, int n_units, int rank, int first_warp)
{
    const int lane = static_cast<int>(ptx::lane_id());
    const int w = static_cast<int>(threadIdx.x / 32) - first_warp;
    const int n_warps = kWaitWarp - first_warp;   // warps first_warp .. kWaitWarp - 1
    const int S = p.n_shards;
    const int n_tiles = p.rs_tiles;
    const size_t row_bytes = static_cast<size_t>(p.N) * 2;
    const size_t shard_bytes = static_cast<size_t>(p.M) * row_bytes;
    for (int t = unit; t < n_tiles; t += n_units) {
        const int o = t / S;
        if (t % S != o % S) continue;               // another CTA (pair) owns output tile o
        for (int s0 = 0; s0 < S; s0 += 32)
            if (warp_wait_lanes(s0 + lane < S ? p.ctrl.slot + o * S + s0 + lane : nullptr, p.gate_seq, p.ctrl, p.seq,
                                p.timeout_ns) < 0)
                return;
        // this CTA's rows of the tile: row block (o / n_nb) * rs_pair + rank
        const int row0 = ((o / p.n_nb) * p.rs_pair + rank) * kTileM;
        const size_t col = static_cast<size_t>(o % p.n_nb) * kTileN * 2 + static_cast<size_t>(lane) * 16;
        const uint8_t* part = static_cast<const uint8_t*>(p.out) + col;
        uint8_t* out = static_cast<uint8_t*>(p.rs_out) + col;
#pragma unroll 1
        for (int r = w * kRsRows; r < kTileM; r += n_warps * kRsRows) {
            // rows r .. r + kRsRows - 1 of the CTA's 128 (kTileM is a multiple of kRsRows)
            float acc[kRsRows][8];
#pragma unroll
            for (int j = 0; j < kRsRows; ++j)
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[j][c] = 0.0f;
            const uint8_t* base = part + static_cast<size_t>(row0 + r) * row_bytes;
#pragma unroll 1
            for (int sb = 0; sb < S; sb += kRsShards) {
                int4 v[kRsShards][kRsRows];
#pragma unroll
                for (int q = 0; q < kRsShards; ++q) {
                    // shards past S re-read the last one (unconditional loads; their sums are skipped)
                    const int sh = min(sb + q, S - 1);
#pragma unroll
                    for (int j = 0; j < kRsRows; ++j)
                        v[q][j] = ptx::ld_v4(reinterpret_cast<const int4*>(base + sh * shard_bytes + j * row_bytes));
                }
#pragma unroll
                for (int q = 0; q < kRsShards; ++q) {
                    if (sb + q >= S) break;
#pragma unroll
                    for (int j = 0; j < kRsRows; ++j) {
                        const uint32_t u[4] = {static_cast<uint32_t>(v[q][j].x), static_cast<uint32_t>(v[q][j].y),
                                               static_cast<uint32_t>(v[q][j].z), static_cast<uint32_t>(v[q][j].w)};
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            acc[j][2 * c] = __fadd_rn(acc[j][2 * c], __uint_as_float(u[c] << 16));
                            acc[j][2 * c + 1] = __fadd_rn(acc[j][2 * c + 1], __uint_as_float(u[c] & 0xffff0000u));
                        }
                    }
                }
            }
            uint8_t* dst = out + static_cast<size_t>(row0 + r) * row_bytes;
#pragma unroll
            for (int j = 0; j < kRsRows; ++j) {
                int4 o4;
                o4.x = static_cast<int>(ptx::pack_bf16x2(acc[j][0], acc[j][1]));
                o4.y = static_cast<int>(ptx::pack_bf16x2(acc[j][2], acc[j][3]));
                o4.z = static_cast<int>(ptx::pack_bf16x2(acc[j][4], acc[j][5]));
                o4.w = static_cast<int>(ptx::pack_bf16x2(acc[j][6], acc[j][7]));
                ptx::st_v4(reinterpret_cast<int4*>(dst + j * row_bytes), o4);
            }
        }
    }
}

__device__ inline void producer(const FusedParams& p, uint8_t* smem, int pid)
{
    const int warp = threadIdx.x / 32;
    const int n_warps = kThreads / 32;
    // consecutive items go to different CTAs (SMs), so the rows of one chunk
    // are copied by many SMs at once
    const int gw = warp * p.n_producers + pid;
    const int n_gw = p.n_producers * n_warps;
    if (threadIdx.x == 0) stat_min(p, kStatProdStartNs, ptx::globaltimer());
    // sources, plan and counters were written by earlier kernels
    ptx::grid_dep_wait();
    seed_counters(p, gw, n_gw, true);
    if (p.mode == kModeReduceScatter) {
        rs_reduce(p);
    } else if (p.producer_mode == 1) {
        if (p.item_rows <= 16) copy_items_staged<1>(p, smem, gw, n_gw);
        else if (p.item_rows == 32) copy_items_staged<2>(p, smem, gw, n_gw);
        else copy_items_staged<4>(p, smem, gw, n_gw);
    } else {
        if (p.item_rows <= 16) copy_items<1>(p, gw, n_gw);
        else if (p.item_rows == 32) copy_items<2>(p, gw, n_gw);
        else copy_items<4>(p, gw, n_gw);
    }
    seed_counters(p, gw, n_gw, false);
    __syncwarp();
    __syncthreads();
    if (threadIdx.x == 0) stat_max(p, kStatProdEndNs, ptx::globaltimer());
}

}  // namespace tovl
