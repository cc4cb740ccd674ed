// fused.cu -- the persistent fused gather/dispatch + GEMM kernel.
//
// One cooperative launch of P producer CTAs and C consumer CTAs, one CTA per
// SM, all co-resident:
//   producers  copy token rows into the gathered (or dispatched) buffer with
//              16-byte vector loads/stores and count them with the
//              single-writer protocol: an acq_rel arrival count per 64-row
//              chunk whose last arrival is elected to release-store the
//              round's sequence number into the chunk's watermark slot
//              (gather), or release reductions into 128-row block counters
//              pre-seeded with the padding count (dispatch) -- "cross-GPU sync
//              protocols on PCIe", sections 3-5;
//   consumers  run a tcgen05 bf16 GEMM over 128x256 output tiles in
//              row-block order; the TMA warp of each consumer gates the rows
//              of a tile on the protocol with acquire polls before loading
//              them.
// Each chunk watermark may be split along K into k_slices sub-watermarks:
// the consumer's minimal release unit is a K-range of a row block, and the
// signal follows it (section 4: signal granularity follows the consumer's
// release unit).  Producers copy in the consumers' traversal order -- first
// wave's row blocks, slice by slice, then the next wave's (section 6, item 3)
// -- so the first tiles start after a fraction of their rows has landed.
// With k_slices = 1 each slot is exactly one 64-row chunk watermark.
// Producers never wait on anyone; consumers wait only on producers, which are
// resident by construction (cooperative launch), and every wait is bounded.
#include <cuda_runtime.h>
#include "ctrl.cuh"
#include "ptx.cuh"
#include "sync.cuh"
#include "launch.cuh"

namespace tovl {

// Instruction descriptor: M=128, N=256, A K-major (gathered rows), B
// MN-major (W is [K][N] with N contiguous).
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kTileM, kTileN, false, true);

__device__ __forceinline__ uint8_t* align1024(uint8_t* p)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return reinterpret_cast<uint8_t*>((a + 1023) & ~static_cast<uintptr_t>(1023));
}

__device__ __forceinline__ void stat_min(const FusedParams& p, int idx, unsigned long long v)
{
    if (p.stats) atomicMin(p.ctrl.stats + idx, v);
}

__device__ __forceinline__ void stat_max(const FusedParams& p, int idx, unsigned long long v)
{
    if (p.stats) atomicMax(p.ctrl.stats + idx, v);
}

// Number of 128-row blocks the consumers traverse this round.
__device__ __forceinline__ int num_row_blocks(const FusedParams& p)
{
    if (p.mode == kModeGather) return (p.M + kTileM - 1) / kTileM;
    return p.meta[1];
}

// K-blocks [kb_begin(s), kb_begin(s+1)) form slice s.
__device__ __forceinline__ int kb_begin(const FusedParams& p, int s)
{
    return s * p.n_kb / p.k_slices;
}

// ============================================================= consumers
struct ConsumerSmem {
    uint8_t* a;          // kStages x [128 rows][128 B]  (A tile, 128B swizzle)
    uint8_t* b;          // kStages x 4 x [64 k-rows][128 B]  (B tile: four 64-column blocks)
    uint64_t* full;      // TMA -> MMA
    uint64_t* empty;     // MMA -> TMA
    uint64_t* tfull;     // MMA -> epilogue (per accumulator)
    uint64_t* tempty;    // epilogue -> MMA
    uint32_t* tmem_slot;
    int* gates_passed;   // gate warp -> TMA warp: number of (tile, slice) gates passed
};

__device__ __forceinline__ ConsumerSmem consumer_smem(uint8_t* smem)
{
    ConsumerSmem s;
    s.a = smem;
    s.b = smem + kStages * kStageA;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    s.full = bars;
    s.empty = bars + kStages;
    s.tfull = bars + 2 * kStages;
    s.tempty = bars + 2 * kStages + 2;
    s.tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 4);
    s.gates_passed = reinterpret_cast<int*>(bars + 2 * kStages + 5);
    return s;
}

__device__ __forceinline__ void trace_put(const FusedParams& p, long long idx, unsigned long long v)
{
    if (p.stats && idx < p.ctrl.trace_cap) p.ctrl.trace[idx] = static_cast<long long>(v);
}

// Gate: the rows of row block mb, K-slice s, are complete this round.
__device__ __forceinline__ unsigned long long gate(const FusedParams& p, int mb, int s)
{
    const int* words[kTileM / kChunkRows];
    int n = 0;
    int target;
    const int S = p.ctrl.n_slices;
    if (p.mode == kModeGather) {
        const int c0 = mb * (kTileM / kChunkRows);
        for (int i = 0; i < kTileM / kChunkRows; ++i)
            if ((c0 + i) * kChunkRows < p.M) words[n++] = p.ctrl.slot + (c0 + i) * S + s;
        target = p.gate_seq;
    } else {
        words[n++] = p.ctrl.rbcnt + mb * S + s;
        target = p.gate_seq * kBlockRows;
    }
    const int r = warp_wait_ge(words, n, target, p.ctrl, p.seq, p.timeout_ns);
    return static_cast<unsigned long long>(r < 0 ? -r : r);
}

// Gate warp: walks the consumer's (tile, slice) schedule ahead of the TMA
// warp, waits for each slice's rows on the protocol (acquire polls of the
// local slots / counters) and hands every passed gate to the TMA warp with a
// CTA-scope release of the running count.  A gate that times out is handed
// on as well, so the pipeline drains; the status word holds the error.
__device__ void consumer_gate(const FusedParams& p, const ConsumerSmem& s, int cid, int n_tiles)
{
    const uint32_t lane = ptx::lane_id();
    unsigned long long polls = 0;
    int passed = 0;
    for (int t = cid; t < n_tiles; t += p.n_consumers) {
        const int mb = t / p.n_nb;
        for (int sl = 0; sl < p.k_slices; ++sl) {
            polls += gate(p, mb, sl);
            ++passed;
            if (lane == 0) {
                ptx::st_release_cta_smem(s.gates_passed, passed);
                trace_put(p, static_cast<long long>(t) * p.k_slices + sl, ptx::globaltimer());
            }
            __syncwarp();
        }
    }
    if (p.stats && lane == 0 && polls) atomicAdd(p.ctrl.stats + kStatGatePolls, polls);
}

// TMA lane: wait until the gate warp has passed gate number `idx` (bounded).
__device__ __forceinline__ bool wait_gate(const FusedParams& p, const ConsumerSmem& s, int idx)
{
    if (ptx::ld_acquire_cta_smem(s.gates_passed) > idx) return true;
    const uint64_t start = ptx::globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (ptx::ld_acquire_cta_smem(s.gates_passed) > idx) return true;
        if ((i & 63) == 0 && ptx::globaltimer() - start > static_cast<uint64_t>(p.pipe_timeout_ns)) {
            record_error(p.ctrl, kErrTimeout);
            return false;
        }
        __nanosleep(20);
    }
}

// TMA warp: per tile and K-slice, wait for the slice's gate, then stream A
// and B k-blocks into the stage ring.  One lane issues everything.
__device__ void consumer_tma(const FusedParams& p, const ConsumerSmem& s, int cid, int n_tiles)
{
    if (ptx::lane_id() != 0) return;
    uint32_t stage = 0, phase = 0;
    int gate_idx = 0;
    for (int t = cid; t < n_tiles; t += p.n_consumers) {
        const int mb = t / p.n_nb;
        const int nb = t % p.n_nb;
        const int brow = (p.mode == kModeDispatch) ? p.blk_expert[mb] * p.K : 0;
        for (int sl = 0; sl < p.k_slices; ++sl, ++gate_idx) {
            if (p.gated) {
                if (!wait_gate(p, s, gate_idx)) return;
                // the rows were written through the generic proxy; order them
                // before this thread's tensor-memory-access (async proxy) reads
                ptx::fence_proxy_async_global();
            }
            {
                const int kb1 = kb_begin(p, sl + 1);
                for (int kb = kb_begin(p, sl); kb < kb1; ++kb) {
                    if (!mbar_wait(&s.empty[stage], phase ^ 1u, p.ctrl, p.pipe_timeout_ns)) return;
                    ptx::mbar_arrive_expect_tx(&s.full[stage], kStageBytes);
                    ptx::tma_load_2d(s.a + stage * kStageA, &p.tmap_a, &s.full[stage], kb * kTileK, mb * kTileM);
                    uint8_t* bdst = s.b + stage * kStageB;
#pragma unroll
                    for (int j = 0; j < kTileN / 64; ++j)
                        ptx::tma_load_2d(bdst + j * (kTileK * 128), &p.tmap_b, &s.full[stage], nb * kTileN + j * 64,
                                         brow + kb * kTileK);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    }
}

// MMA warp: one lane issues tcgen05.mma into a double-buffered TMEM
// accumulator (2 x 256 fp32 columns).
__device__ void consumer_mma(const FusedParams& p, const ConsumerSmem& s, int cid, int n_tiles, uint32_t tmem_base)
{
    if (ptx::lane_id() != 0) return;
    uint32_t stage = 0, phase = 0;
    int local = 0;
    for (int t = cid; t < n_tiles; t += p.n_consumers, ++local) {
        const uint32_t acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!mbar_wait(&s.tempty[acc], acc_phase ^ 1u, p.ctrl, p.pipe_timeout_ns)) return;
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + acc * kTileN;
        for (int kb = 0; kb < p.n_kb; ++kb) {
            if (!mbar_wait(&s.full[stage], phase, p.ctrl, p.pipe_timeout_ns)) return;
            ptx::tc_fence_after();
            const uint32_t a0 = ptx::smem_u32(s.a + stage * kStageA);
            const uint32_t b0 = ptx::smem_u32(s.b + stage * kStageB);
#pragma unroll
            for (int k = 0; k < kTileK / kUmmaK; ++k) {
                // A: K-major, 128B swizzle; +32 B per 16-element k step inside the swizzle row;
                //    8-row groups 1024 B apart.
                const uint64_t ad = ptx::smem_desc_sw128(a0 + k * 32, 16, 1024);
                // B: MN-major, 128B swizzle; +2048 B per 16 k-rows; 8-k-row groups 1024 B apart;
                //    64-column blocks 8 KB apart.
                const uint64_t bd = ptx::smem_desc_sw128(b0 + k * 2048, kTileK * 128, 1024);
                ptx::umma_bf16(d, ad, bd, kIdesc, (kb | k) != 0);
            }
            ptx::umma_commit(&s.empty[stage]);
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        ptx::umma_commit(&s.tfull[acc]);
    }
}

// Epilogue warps: TMEM -> registers -> bf16 (round to nearest even) -> out.
// Warp w reads TMEM lane quarter w % 4 (the quarter its position allows) and
// one half of the 256 accumulator columns.
__device__ void consumer_epilogue(const FusedParams& p, const ConsumerSmem& s, int cid, int n_tiles,
                                  uint32_t tmem_base, int valid_rows)
{
    const int warp = threadIdx.x / 32;
    const uint32_t lane = ptx::lane_id();
    const int q = warp & 3;
    const int half = (warp - kEpiWarp0) / 4;
    const int row_in_tile = q * 32 + static_cast<int>(lane);
    uint16_t* out = static_cast<uint16_t*>(p.out);
    int local = 0;
    for (int t = cid; t < n_tiles; t += p.n_consumers, ++local) {
        const int mb = t / p.n_nb;
        const int nb = t % p.n_nb;
        const uint32_t acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        const bool arrived = mbar_wait(&s.tfull[acc], acc_phase, p.ctrl, p.pipe_timeout_ns);
        if (!__all_sync(0xffffffffu, arrived)) return;
        ptx::tc_fence_after();
        const int row = mb * kTileM + row_in_tile;
        const bool ok = row < valid_rows;
        const int col0 = half * (kTileN / 2);
        uint4* dst = reinterpret_cast<uint4*>(out + static_cast<size_t>(row) * p.N + nb * kTileN + col0);
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kTileN + col0;
#pragma unroll 1
        for (int c = 0; c < kTileN / 2 / 32; ++c) {
            uint32_t r[32];
            ptx::tmem_ld_32x32b_x32(taddr + c * 32, r);
            ptx::tmem_ld_wait();
            if (ok) {
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    uint4 w;
                    w.x = ptx::pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
                    w.y = ptx::pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
                    w.z = ptx::pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
                    w.w = ptx::pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
                    dst[c * 4 + v] = w;
                }
            }
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(&s.tempty[acc]);
        if (p.stats && lane == 0) {
            const long long idx = static_cast<long long>(p.trace_tiles) * p.k_slices + t;
            if (idx < p.ctrl.trace_cap)
                atomicMax(reinterpret_cast<unsigned long long*>(p.ctrl.trace + idx), ptx::globaltimer());
        }
    }
}

__device__ void consumer(const FusedParams& p, uint8_t* smem, int cid)
{
    const int warp = threadIdx.x / 32;
    const ConsumerSmem s = consumer_smem(smem);
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            ptx::mbar_init(&s.full[i], 1);
            ptx::mbar_init(&s.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&s.tfull[i], 1);
            ptx::mbar_init(&s.tempty[i], kEpiWarps * 32);
        }
        *s.gates_passed = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&p.tmap_a);
        ptx::prefetch_tmap(&p.tmap_b);
        stat_min(p, kStatConsStartNs, ptx::globaltimer());
    }
    if (warp == 1) {
        ptx::tmem_alloc(s.tmem_slot, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *s.tmem_slot;

    const int n_tiles = num_row_blocks(p) * p.n_nb;
    const int valid_rows = (p.mode == kModeGather) ? p.M : p.meta[0];
    if (warp == 0) consumer_tma(p, s, cid, n_tiles);
    else if (warp == 1) consumer_mma(p, s, cid, n_tiles, tmem_base);
    else if (warp < kEpiWarp0 + kEpiWarps) consumer_epilogue(p, s, cid, n_tiles, tmem_base, valid_rows);
    else if (warp == kGateWarp && p.gated) consumer_gate(p, s, cid, n_tiles);
    __syncwarp();

    // teardown: full-CTA barrier 0, after every role has finished
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
    if (threadIdx.x == 0) stat_max(p, kStatConsEndNs, ptx::globaltimer());
}

// ============================================================= producers
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
    const int gw = pid * n_warps + warp;
    const int n_gw = p.n_producers * n_warps;
    if (threadIdx.x == 0) stat_min(p, kStatProdStartNs, ptx::globaltimer());
    seed_counters(p, gw, n_gw, true);

    const uint8_t** tbl = reinterpret_cast<const uint8_t**>(smem) + warp * 64;   // row-source table per warp
    const int n_blocks = num_row_blocks(p);
    const int n_items = n_blocks * p.k_slices * (kBlockRows / p.item_rows);
    const int S = p.ctrl.n_slices;
    // Items of the consumers' first wave are released one by one (their
    // consumers are already waiting); later items in batches, which saves
    // release fences.  Lane j < kReleaseBatch holds the batch's j-th item.
    const int first_wave_items = p.wave_blocks * p.k_slices * (kBlockRows / p.item_rows);
    int pend_counter = 0, pend_n = 0, n_pend = 0;
    for (int i = gw; i < n_items; i += n_gw) {
        const Item it = decode_item(p, i, n_blocks);
        const int n = copy_item(p, it, tbl);
        const int counter = (p.mode == kModeGather) ? (it.r0 / kChunkRows) * S + it.s : it.mb * S + it.s;
        if (static_cast<int>(lane) == n_pend) {
            pend_counter = counter;
            pend_n = n;
        }
        if (++n_pend == kReleaseBatch || i < first_wave_items) {
            // the copies above happen-before every lane's release below
            __syncwarp();
            if (static_cast<int>(lane) < n_pend && pend_n > 0) item_done(p, pend_counter, pend_n);
            n_pend = 0;
        }
    }
    __syncwarp();
    if (static_cast<int>(lane) < n_pend && pend_n > 0) item_done(p, pend_counter, pend_n);
    __syncwarp();
    seed_counters(p, gw, n_gw, false);
    __syncwarp();
    __syncthreads();
    if (threadIdx.x == 0) stat_max(p, kStatProdEndNs, ptx::globaltimer());
}

// ============================================================= kernel
__global__ void __launch_bounds__(kThreads, 1) fused_kernel(const __grid_constant__ FusedParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    if (static_cast<int>(blockIdx.x) < p.n_producers) producer(p, smem, blockIdx.x);
    else consumer(p, smem, blockIdx.x - p.n_producers);
}

cudaError_t launch_fused(const FusedParams& p, cudaStream_t stream, bool cooperative)
{
    const int grid = p.n_producers + p.n_consumers;
    if (grid <= 0) return cudaSuccess;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(grid);
    lc.blockDim = dim3(kThreads);
    lc.dynamicSmemBytes = kSmemBytes;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = cooperative ? 1 : 0;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, fused_kernel, p);
}

cudaError_t prepare_fused()
{
    return cudaFuncSetAttribute(fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

int fused_max_active_per_sm()
{
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fused_kernel, kThreads, kSmemBytes) != cudaSuccess) return 0;
    return n;
}

}  // namespace tovl
