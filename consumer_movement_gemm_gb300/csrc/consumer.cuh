// consumer.cuh -- consumer CTAs of the fused kernel: gated tcgen05 GEMM.
//
// A consumer CTA (or a pair of CTAs in a cluster, PAIR = 2) computes output
// tiles in row-block order, the producers' order ("cross-GPU sync protocols
// on PCIe", section 6 item 3).  Warp roles:
//   warp 0      TMA: per tile and K-slice, waits for the slice's gate, then
//               streams A (gathered rows, one box per k-block) and B
//               (weights, one 3-D box of kWBlocks 64-column blocks) into a
//               ring of shared-memory stages
//   warp 1      MMA: one lane issues tcgen05.mma into a double-buffered TMEM
//               accumulator (2 x 256 fp32 columns)
//   warps 2-9   epilogue: TMEM -> registers -> bf16 (nearest even) -> out
//   warp 10     gate: polls the protocol (acquire loads of local slots /
//               counters, ballot) ahead of the TMA warp and hands each
//               passed gate over through shared memory
//   warps 11-14 idle, or the embedded producers' copy warps (launches
//               without producer CTAs), or (with warp 10) the owners'
//               reducers of a reduce-scatter with option 19
//   warp 15     stage waiter: observes each stage's full barrier and hands
//               the stage to the MMA warp on a named barrier (fixed
//               schedule; the dynamic schedule's MMA lane waits itself)
// PAIR = 1: 128x256 tiles, stage = A 16 KB + B 32 KB, 4 stages.
// PAIR = 2: 256x256 tiles per CTA pair (cta_group::2).  Each CTA stages its
// own 128 rows of A and 128 of B's 256 columns (stage 32 KB, 5 stages beside
// producer CTAs, 6 without).  A dispatch with embedded producers takes
// 256x512 tiles where N allows (NW = 2): two N = 256 MMAs per k-step into
// one 512-column accumulator, each CTA staging A 16 KB and 128 of each
// half's 256 columns (one 4-D weight box) per k-block, 4 stages.  The pair's
// first CTA issues the MMAs, which read A and B halves from both CTAs and
// accumulate each CTA's rows in its own TMEM.  Both CTAs' TMA loads are
// counted on the first CTA's "full" barriers; MMA completion is multicast to
// both CTAs; each CTA's epilogue warps release the accumulator on the first
// CTA's "tmem empty" barrier.
#pragma once
#include "common.cuh"
#include "ctrl.cuh"
#include "ptx.cuh"
#include "sync.cuh"
#include "producer.cuh"

namespace tovl {

// NW = 256-column MMAs per k-step: 1 for 256-column tiles (double-buffered
// accumulator), 2 for 512-column CTA-pair tiles (one accumulator of all 512
// TMEM columns; the weights as one 4-D box per k-block).
template <int PAIR, int ST = stages_for(PAIR), int NW = 1>
struct Tile {
    static constexpr int kStages = ST;
    static constexpr int kStageA = kTileM * kTileK * 2;               // 16 KB
    static constexpr int kStageB = kTileK * kTileN * NW * 2 / PAIR;   // this CTA's B columns
    static constexpr int kStageBytes = kStageA + kStageB;
    static constexpr int kBBoxes = kTileN * NW / 64 / PAIR;           // 64-column blocks per stage
    static constexpr int kCols = kTileN * NW;                         // output columns of a tile
    // M = 128 * PAIR, N = 256, A K-major, B MN-major (W is [K][N], N contiguous)
    static constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kTileM * PAIR, kTileN, false, true);
    static_assert(NW == 1 || PAIR == 2, "512-column tiles are CTA-pair tiles");
    static_assert(kStages * kStageBytes + kEpiWarps * kEpiBufBytes * NW + 1024 <= smem_for(PAIR, ST, NW),
                  "stages and epilogue buffers must fit the dynamic shared memory");
    static_assert(smem_for(PAIR, ST, NW) <= 227 * 1024, "at most 227 KB of shared memory per CTA");
};

template <int PAIR>
struct ConsumerSmem {
    uint8_t* a;          // kStages x [128 rows][128 B]  (A tile, 128B swizzle)
    uint8_t* b;          // kStages x kBBoxes x [64 k-rows][128 B]  (this CTA's B columns)
    uint8_t* epi;        // kEpiWarps x [32 rows][64 B] output staging (64B swizzle)
    uint64_t* full;      // TMA -> MMA (in the pair's first CTA: counts both CTAs' bytes)
    uint64_t* empty;     // MMA -> TMA
    uint64_t* tfull;     // MMA -> epilogue (per accumulator)
    uint64_t* tempty;    // epilogue -> MMA (in the pair's first CTA: both CTAs' warps)
    uint32_t* tmem_slot;
    int* gates_passed;   // gate warp -> TMA warp: number of (tile, slice) gates passed
    int* ring;           // dynamic schedule: kRing tile indices handed to the other roles (-1 = no more)
    int* ring_head;      // entries published
    int* epi_started;    // epilogue warps' tile starts (kEpiWarps per tile): ring entries that are free
    int* tma_done;       // k-blocks whose loads the TMA warp has issued (dynamic schedule)
};

constexpr int kRing = 8;

template <int PAIR, int ST = stages_for(PAIR), int NW = 1>
__device__ __forceinline__ ConsumerSmem<PAIR> consumer_smem(uint8_t* smem)
{
    using T = Tile<PAIR, ST, NW>;
    ConsumerSmem<PAIR> s;
    s.a = smem;
    s.b = smem + T::kStages * T::kStageA;
    s.epi = smem + T::kStages * T::kStageBytes;   // 1024-byte aligned: stages are multiples of 1 KB
    uint64_t* bars = reinterpret_cast<uint64_t*>(s.epi + kEpiWarps * kEpiBufBytes * NW);
    s.full = bars;
    s.empty = bars + T::kStages;
    s.tfull = bars + 2 * T::kStages;
    s.tempty = bars + 2 * T::kStages + 2;
    s.tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * T::kStages + 4);
    s.gates_passed = reinterpret_cast<int*>(bars + 2 * T::kStages + 5);
    s.ring = reinterpret_cast<int*>(bars + 2 * T::kStages + 6);
    s.ring_head = s.ring + kRing;
    s.epi_started = s.ring_head + 1;
    s.tma_done = s.ring_head + 2;
    return s;
}

// Tiles of this consumer unit (a CTA, or a CTA pair): unit u of n_units
// takes tiles u, u + n_units, ...; a tile covers PAIR consecutive row blocks
// and one 256-column block.  For a reduce-scatter round tile t is shard
// t % S's partial of output tile t / S, so the S partials of one output tile
// are computed side by side.
template <int PAIR>
struct Schedule {
    int unit, n_units, n_tiles;
    uint32_t rank;
    __device__ int out_tile(const FusedParams& p, int t) const
    {
        return p.mode == kModeReduceScatter ? t / p.n_shards : t;
    }
    __device__ int shard(const FusedParams& p, int t) const { return p.mode == kModeReduceScatter ? t % p.n_shards : 0; }
    // 128-row dispatch segments on CTA pairs: tile row r is the plan's pair
    // tile r (its first block and the next); the next block is a phantom
    // when it lies past the segment: computed with the segment's weights,
    // never gated and never stored
    __device__ int pair_entry(const FusedParams& p, int t) const { return p.pair_tab[1 + out_tile(p, t) / p.n_nb]; }
    __device__ int row_block(const FusedParams& p, int t) const
    {
        if (PAIR == 2 && p.pair_tab) return (pair_entry(p, t) >> 1) + static_cast<int>(rank);
        return (out_tile(p, t) / p.n_nb) * PAIR + static_cast<int>(rank);
    }
    // the row block whose expert's weights the tile multiplies (the pair's first)
    __device__ int expert_block(const FusedParams& p, int t) const
    {
        if (PAIR == 2 && p.pair_tab) return pair_entry(p, t) >> 1;
        return (out_tile(p, t) / p.n_nb) * PAIR;
    }
    __device__ bool phantom(const FusedParams& p, int t) const
    {
        return PAIR == 2 && p.pair_tab && rank == 1 && (pair_entry(p, t) & 1) == 0;
    }
    __device__ int col_block(const FusedParams& p, int t) const { return out_tile(p, t) % p.n_nb; }
    // first row of this CTA's part of the tile in the A and output tensors
    // (reduce-scatter: shard s's rows start at s * M)
    __device__ int a_row(const FusedParams& p, int t) const
    {
        return shard(p, t) * (p.mode == kModeReduceScatter ? p.M : 0) + row_block(p, t) * kTileM;
    }
};

template <int PAIR>
__device__ __forceinline__ Schedule<PAIR> make_schedule(const FusedParams& p, int cid)
{
    Schedule<PAIR> sc;
    sc.rank = PAIR == 2 ? ptx::cluster_ctarank() : 0u;
    sc.unit = cid / PAIR;
    sc.n_units = p.n_consumers / PAIR;
    sc.n_tiles = (num_row_blocks(p) + PAIR - 1) / PAIR * p.n_nb * (p.mode == kModeReduceScatter ? p.n_shards : 1);
    if (PAIR == 2 && p.pair_tab) sc.n_tiles = p.pair_tab[0] * p.n_nb;
    return sc;
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

// Gate warp: walks this CTA's (tile, slice) schedule ahead of the TMA warp,
// waits for each slice's rows on the protocol and hands every passed gate to
// the TMA warp with a CTA-scope release of the running count.  A gate that
// times out is handed on as well, so the pipeline drains; the status word
// holds the error.
template <int PAIR>
__device__ void consumer_gate(const FusedParams& p, const ConsumerSmem<PAIR>& s, const Schedule<PAIR>& sc)
{
    const uint32_t lane = ptx::lane_id();
    unsigned long long polls = 0;
    int passed = 0;
    for (int t = sc.unit; t < sc.n_tiles; t += sc.n_units) {
        const int mb = sc.row_block(p, t);
        const bool phantom = sc.phantom(p, t);
        for (int sl = 0; sl < p.k_slices; ++sl) {
            if (!phantom) polls += gate(p, mb, sl);
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

// Weight (B) cursor of the TMA lane.  B does not depend on the producers, so
// its k-blocks are loaded ahead of the gate: a stage's B boxes are issued (and
// the stage's full barrier armed for A + B bytes) as soon as the stage is
// free, and the stage's A box follows once the slice's gate has passed.
template <int PAIR>
struct BCursor {
    int t, kb, brow, n0;      // next k-block to load: tile, k-block, B row base, B column base
    int issued;               // stages armed so far
    uint32_t stage, phase;
    uint64_t pol;             // L2 policy of the weight loads
};

template <int PAIR, int NW = 1>
__device__ __forceinline__ void b_tile(const FusedParams& p, const Schedule<PAIR>& sc, BCursor<PAIR>& b)
{
    if (b.t >= sc.n_tiles) return;
    const int mb = sc.expert_block(p, b.t);
    b.brow = (p.mode == kModeDispatch) ? p.blk_expert[mb] * p.K
           : (p.mode == kModeReduceScatter) ? sc.shard(p, b.t) * p.K : 0;
    b.n0 = sc.col_block(p, b.t) * kTileN * NW + static_cast<int>(sc.rank) * (kTileN / PAIR);
}

// Arm the cursor's stage and issue its B boxes (the stage must be free).
template <int PAIR, int ST, int NW = 1>
__device__ __forceinline__ void b_issue(const FusedParams& p, const ConsumerSmem<PAIR>& s, const Schedule<PAIR>& sc,
                                        BCursor<PAIR>& b)
{
    using T = Tile<PAIR, ST, NW>;
    uint8_t* bdst = s.b + b.stage * T::kStageB;
    // one 3-D load per kWBlocks 64-column blocks (measured: each tensor-load
    // instruction stalls the MMA stream, two 2-D boxes per k-block cost 9.5
    // clocks per pair MMA more than one 3-D box)
    static_assert(T::kBBoxes % kWBlocks == 0, "whole weight loads per stage");
    if (PAIR == 1) {
        ptx::mbar_arrive_expect_tx(&s.full[b.stage], T::kStageBytes);
#pragma unroll
        for (int j = 0; j < T::kBBoxes; j += kWBlocks)
            ptx::tma_load_3d_hint(bdst + j * (kTileK * 128), &p.tmap_b, &s.full[b.stage], 0, b.brow + b.kb * kTileK,
                                  b.n0 / 64 + j, b.pol);
    } else if (NW == 2) {
        // 512-column tiles: this CTA's 128 columns of each of the tile's two
        // 256-column halves in one 4-D box ([N/256][4][rows][64] view, box
        // 64 x 64 x 2 x 2): block z of half h lands h * 16 KB + z * 8 KB in
        if (sc.rank == 0) ptx::mbar_arrive_expect_tx(&s.full[b.stage], PAIR * T::kStageBytes);
        const uint32_t bar0 = ptx::mapa_shared(ptx::smem_u32(&s.full[b.stage]), 0);
        ptx::tma_load_4d_pair_hint(bdst, &p.tmap_b, bar0, 0, b.brow + b.kb * kTileK, (b.n0 % kTileN) / 64,
                                   b.n0 / kTileN, b.pol);
    } else {
        // both CTAs' bytes are counted on the first CTA's barrier
        if (sc.rank == 0) ptx::mbar_arrive_expect_tx(&s.full[b.stage], PAIR * T::kStageBytes);
        const uint32_t bar0 = ptx::mapa_shared(ptx::smem_u32(&s.full[b.stage]), 0);
#pragma unroll
        for (int j = 0; j < T::kBBoxes; j += kWBlocks)
            ptx::tma_load_3d_pair_hint(bdst + j * (kTileK * 128), &p.tmap_b, bar0, 0, b.brow + b.kb * kTileK,
                                       b.n0 / 64 + j, b.pol);
    }
    ++b.issued;
    if (++b.stage == T::kStages) {
        b.stage = 0;
        b.phase ^= 1u;
    }
    if (++b.kb == p.n_kb) {
        b.kb = 0;
        b.t += sc.n_units;
        b_tile<PAIR, NW>(p, sc, b);
    }
}

// Arm stages until the cursor is `ahead` stages past `a_count` (blocking on
// free stages only when `block`).  Returns false on a pipeline timeout.
template <int PAIR, int ST, int NW = 1>
__device__ __forceinline__ bool b_run(const FusedParams& p, const ConsumerSmem<PAIR>& s, const Schedule<PAIR>& sc,
                                      BCursor<PAIR>& b, int upto, bool block)
{
    while (b.issued < upto && b.t < sc.n_tiles) {
        if (block) {
            if (!mbar_wait(&s.empty[b.stage], b.phase ^ 1u, p.ctrl, p.pipe_timeout_ns)) return false;
        } else if (!ptx::mbar_try_wait(&s.empty[b.stage], b.phase ^ 1u)) {
            return true;
        }
        b_issue<PAIR, ST, NW>(p, s, sc, b);
    }
    return true;
}

// TMA lane: wait until the gate warp has passed gate number `idx` (bounded),
// arming free stages with B meanwhile.
template <int PAIR, int ST, int NW = 1>
__device__ __forceinline__ bool wait_gate(const FusedParams& p, const ConsumerSmem<PAIR>& s, const Schedule<PAIR>& sc,
                                          BCursor<PAIR>& b, int a_count, int idx)
{
    using T = Tile<PAIR, ST, NW>;
    if (ptx::ld_acquire_cta_smem(s.gates_passed) > idx) return true;
    const uint64_t start = ptx::globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (!b_run<PAIR, ST, NW>(p, s, sc, b, a_count + T::kStages, false)) return false;
        if (ptx::ld_acquire_cta_smem(s.gates_passed) > idx) return true;
        if ((i & 63) == 0 && ptx::globaltimer() - start > static_cast<uint64_t>(p.pipe_timeout_ns)) {
            record_error(p.ctrl, kErrTimeout);
            return false;
        }
        __nanosleep(20);
    }
}

// TMA warp: per tile and K-slice, wait for the slice's gate, then stream the
// slice's A k-blocks into stages whose B the cursor above has already
// loaded.  One lane issues everything.
template <int PAIR, int ST, int NW = 1>
__device__ void consumer_tma(const FusedParams& p, const ConsumerSmem<PAIR>& s, const Schedule<PAIR>& sc)
{
    using T = Tile<PAIR, ST, NW>;
    if (ptx::lane_id() != 0) return;
    BCursor<PAIR> b;
    b.t = sc.unit;
    b.kb = 0;
    b.issued = 0;
    b.stage = 0;
    b.phase = 0;
    b.pol = stream_policy(p, kHintBLast, 0);
    const uint64_t pol_a = stream_policy(p, 0, kHintAFirst);
    b_tile<PAIR, NW>(p, sc, b);
    uint32_t stage = 0;
    int a_count = 0;
    int gate_idx = 0;
    for (int t = sc.unit; t < sc.n_tiles; t += sc.n_units) {
        const int arow = sc.a_row(p, t);
        for (int sl = 0; sl < p.k_slices; ++sl, ++gate_idx) {
            if (p.gated) {
                if (!wait_gate<PAIR, ST, NW>(p, s, sc, b, a_count, gate_idx)) return;
                // the rows were written through the generic proxy; order them
                // before this thread's tensor-memory-access (async proxy) reads
                ptx::fence_proxy_async_global();
            }
            const int kb1 = kb_begin(p, sl + 1);
            for (int kb = kb_begin(p, sl); kb < kb1; ++kb) {
                // this k-block's stage is armed and holds (or receives) its B
                if (!b_run<PAIR, ST, NW>(p, s, sc, b, a_count + 1, true)) return;
                uint8_t* adst = s.a + stage * T::kStageA;
                if (PAIR == 1) {
                    ptx::tma_load_2d_hint(adst, &p.tmap_a, &s.full[stage], kb * kTileK, arow, pol_a);
                } else {
                    const uint32_t bar0 = ptx::mapa_shared(ptx::smem_u32(&s.full[stage]), 0);
                    ptx::tma_load_2d_pair_hint(adst, &p.tmap_a, bar0, kb * kTileK, arow, pol_a);
                }
                ++a_count;
                if (++stage == T::kStages) stage = 0;
            }
        }
    }
}

// MMA warp (of the pair's first CTA): lane 0 issues the MMAs.  The stages'
// full barriers are observed by the stage waiter warp, which hands each
// stage over on named barrier kStageBar0 + stage; the whole MMA warp takes
// that barrier.  An mbarrier wait on the issuing thread itself stalls the
// MMA stream even when the barrier has long completed (measured with pair
// MMAs over five rotating stages: 128.7 clocks per MMA with no waits, 139.0
// with one already-complete wait per k-block; 141.5 in the full handshake
// against 129.6 with the hand-off).
template <int PAIR, int ST, int NW = 1>
__device__ void consumer_mma(const FusedParams& p, const ConsumerSmem<PAIR>& s, const Schedule<PAIR>& sc,
                             uint32_t tmem_base)
{
    using T = Tile<PAIR, ST, NW>;
    if (sc.rank != 0) return;
    const bool lead = ptx::lane_id() == 0;
    uint32_t stage = 0;
    int local = 0;
    for (int t = sc.unit; t < sc.n_tiles; t += sc.n_units, ++local) {
        // two accumulators used in turn, or (512-column tiles) one
        const uint32_t acc = NW == 1 ? (local & 1) : 0;
        const uint32_t acc_phase = NW == 1 ? ((local >> 1) & 1) : (local & 1);
        if (lead) {
            // a timeout is recorded in the status word; the loop goes on, so
            // every stage hand-off of the waiter is still taken
            mbar_wait(&s.tempty[acc], acc_phase ^ 1u, p.ctrl, p.pipe_timeout_ns);
            ptx::tc_fence_after();
        }
        __syncwarp();
        const uint32_t d = tmem_base + acc * kTileN;
        for (int kb = 0; kb < p.n_kb; ++kb) {
            // the stage's TMA bytes have landed: the waiter observed its full
            // barrier (the barrier's transaction count) and arrived here; the
            // MMAs below read the stage through the async proxy.  No tcgen05
            // thread-sync fence: measured, it costs 14 clocks per MMA
            ptx::bar_sync_aligned(kStageBar0 + static_cast<int>(stage), kStageBarThreads);
            if (lead) {
                const uint32_t a0 = ptx::smem_u32(s.a + stage * T::kStageA);
                const uint32_t b0 = ptx::smem_u32(s.b + stage * T::kStageB);
#pragma unroll
                for (int k = 0; k < kTileK / kUmmaK; ++k) {
                    // A: K-major, 128B swizzle; +32 B per 16-element k step inside
                    //    the swizzle row; 8-row groups 1024 B apart.
                    const uint64_t ad = ptx::smem_desc_sw128(a0 + k * 32, 16, 1024);
                    // B: MN-major, 128B swizzle; +2048 B per 16 k-rows; 8-k-row
                    //    groups 1024 B apart; 64-column blocks 8 KB apart.
                    //    A 512-column tile's second half starts 16 KB in and
                    //    accumulates into TMEM columns 256-511.
#pragma unroll
                    for (int h = 0; h < NW; ++h) {
                        const uint64_t bd =
                            ptx::smem_desc_sw128(b0 + h * (T::kStageB / NW) + k * 2048, kTileK * 128, 1024);
                        if (PAIR == 1) ptx::umma_bf16(d, ad, bd, T::kIdesc, (kb | k) != 0);
                        else ptx::umma_bf16_pair(d + h * kTileN, ad, bd, T::kIdesc, (kb | k) != 0);
                    }
                }
                if (PAIR == 1) ptx::umma_commit(&s.empty[stage]);
                else ptx::umma_commit_pair(&s.empty[stage], 0x3);
            }
            __syncwarp();
            if (++stage == T::kStages) stage = 0;
        }
        if (lead) {
            if (PAIR == 1) ptx::umma_commit(&s.tfull[acc]);
            else ptx::umma_commit_pair(&s.tfull[acc], 0x3);
        }
        __syncwarp();
    }
}

// Stage waiter warp (of the pair's first CTA): walks the MMA warp's k-block
// sequence, lane 0 waits for each stage's full barrier, and the warp arrives
// on the stage's named barrier.  A stage is refilled only after the MMA
// warp's commit for its previous k-block, which follows the MMA warp's wait
// on the same barrier, so no barrier id gets a second arrival before the MMA
// warp has taken the first.  After a timeout lane 0 stops waiting but the
// warp keeps arriving: the MMA warp never blocks on a named barrier.
template <int PAIR, int ST>
__device__ void consumer_stage_waiter(const FusedParams& p, const ConsumerSmem<PAIR>& s, const Schedule<PAIR>& sc)
{
    using T = Tile<PAIR, ST>;
    if (sc.rank != 0) return;
    const bool lead = ptx::lane_id() == 0;
    bool ok = true;
    uint32_t stage = 0, phase = 0;
    for (int t = sc.unit; t < sc.n_tiles; t += sc.n_units) {
        for (int kb = 0; kb < p.n_kb; ++kb) {
            if (lead && ok) ok = mbar_wait(&s.full[stage], phase, p.ctrl, p.pipe_timeout_ns);
            __syncwarp();
            ptx::bar_arrive_aligned(kStageBar0 + static_cast<int>(stage), kStageBarThreads);
            if (++stage == T::kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

// One 32 x 32 box of accumulator values (this lane's row, 32 columns) to the
// output through the warp's staging buffer and coalesced 16-byte stores: four
// lanes cover a row's 64 bytes.
__device__ __forceinline__ void gstore_box(const FusedParams& p, uint32_t row_addr, uint32_t buf_addr, uint32_t swz,
                                           uint32_t lane, int row0, int col, const uint32_t (&r)[32])
{
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const uint32_t chunk = static_cast<uint32_t>(v) ^ swz;
        ptx::st_shared_v4(row_addr + chunk * 16,
                          ptx::pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1])),
                          ptx::pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3])),
                          ptx::pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5])),
                          ptx::pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7])));
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int rr = static_cast<int>(lane >> 2) + 8 * i;
        const uint32_t chunk = (lane & 3u) ^ ((static_cast<uint32_t>(rr) >> 1) & 3u);
        const int4 v = ptx::ld_shared_v4(buf_addr + static_cast<uint32_t>(rr) * (kEpiBoxCols * 2) + chunk * 16);
        const int row = row0 + rr;
        if (row < p.out_rows)
            ptx::st_v4(reinterpret_cast<int4*>(static_cast<uint8_t*>(p.out) + (static_cast<size_t>(row) * p.N + col) * 2) +
                           (lane & 3u),
                       v);
    }
    __syncwarp();   // the buffer is read before the next box overwrites it
}

// Epilogue warps: TMEM -> registers -> bf16 (round to nearest even) ->
// shared memory -> TMA tensor store.  Warp w reads TMEM lane quarter w % 4
// (the quarter its position allows), i.e. 32 output rows, and one half of
// the 256 accumulator columns, as four 32 x 32 boxes.  A box is written into
// the warp's 2 KB buffer in the 64-byte swizzled layout the store's tensor
// map expects (16-byte chunk j of 64-byte row r at chunk j ^ ((r / 2) % 4):
// the eight rows a quarter-warp writes hit distinct banks), then one lane
// stores it; rows past the output's extent (the ragged tail of M) are
// clipped by the store.  Reduce-scatter partial tiles instead leave the
// buffer through the warp's own 16-byte stores (their epilogues come every
// few microseconds, and a tensor store holds its buffer for about a
// microsecond).  The accumulator is released as soon as its last columns are
// in registers.
template <int PAIR, int NW = 1>
__device__ void consumer_epilogue(const FusedParams& p, const ConsumerSmem<PAIR>& s, const Schedule<PAIR>& sc,
                                  uint32_t tmem_base)
{
    // this warp's columns of a tile: half `half` of kCols, kBoxes boxes;
    // 512-column tiles (an exposed drain: no second accumulator) stage their
    // boxes in NW buffers used in turn
    constexpr int kCols = kTileN * NW;
    constexpr int kBoxes = kCols / 2 / kEpiBoxCols;
    const int warp = threadIdx.x / 32;
    const uint32_t lane = ptx::lane_id();
    const int q = warp & 3;
    const int half = (warp - kEpiWarp0) / 4;
    const uint8_t* buf = s.epi + (warp - kEpiWarp0) * kEpiBufBytes * NW;
    const uint32_t row_addr = ptx::smem_u32(buf) + lane * (kEpiBoxCols * 2);
    const uint32_t swz = (lane >> 1) & 3u;
    const uint64_t pol_out = stream_policy(p, 0, kHintOutFirst);
    // reduce-scatter tiles are short (K / S deep) and published one by one:
    // their boxes leave shared memory through this warp's own coalesced
    // stores, so no box waits for a tensor store to finish reading its buffer
    const bool gstore = p.mode == kModeReduceScatter;
    const uint32_t buf_addr = ptx::smem_u32(buf);
    int local = 0;
    for (int t = sc.unit; t < sc.n_tiles; t += sc.n_units, ++local) {
        const int arow = sc.a_row(p, t);
        const int nb = sc.col_block(p, t);
        const uint32_t acc = NW == 1 ? (local & 1) : 0;
        const uint32_t acc_phase = NW == 1 ? ((local >> 1) & 1) : (local & 1);
        const bool arrived = mbar_wait(&s.tfull[acc], acc_phase, p.ctrl, p.pipe_timeout_ns);
        if (!__all_sync(0xffffffffu, arrived)) break;
        ptx::tc_fence_after();
        if (p.stats && lane == 0) {
            const long long idx = static_cast<long long>(p.trace_tiles) * (p.k_slices + 1) + t;
            if (idx < p.ctrl.trace_cap)
                atomicMax(reinterpret_cast<unsigned long long*>(p.ctrl.trace + idx), ptx::globaltimer());
        }
        if (sc.phantom(p, t)) {
            // a phantom half (rows past the segment): nothing is stored;
            // the accumulator goes straight back to the MMA warp
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_u32(&s.tempty[acc]), 0));
            continue;
        }
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kTileN + half * (kCols / 2);
        if (NW == 1 && gstore) {
            // two boxes' accumulator loads in flight per wait
            const int col0 = nb * kTileN + half * (kTileN / 2);
#pragma unroll
            for (int b2 = 0; b2 < kTileN / 2 / kEpiBoxCols; b2 += 2) {
                uint32_t r0[32], r1[32];
                ptx::tmem_ld_32x32b_x32(taddr + b2 * kEpiBoxCols, r0);
                ptx::tmem_ld_32x32b_x32(taddr + (b2 + 1) * kEpiBoxCols, r1);
                ptx::tmem_ld_wait();
                if (b2 + 2 == kTileN / 2 / kEpiBoxCols) {
                    // this warp's reads of the accumulator are done: one arrival per warp
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (PAIR == 1) ptx::mbar_arrive(&s.tempty[acc]);
                        else ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_u32(&s.tempty[acc]), 0));
                    }
                }
                gstore_box(p, row_addr, buf_addr, swz, lane, arow + q * 32, col0 + b2 * kEpiBoxCols, r0);
                gstore_box(p, row_addr, buf_addr, swz, lane, arow + q * 32, col0 + (b2 + 1) * kEpiBoxCols, r1);
            }
        }
#pragma unroll 1
        for (int bx = 0; bx < ((NW == 1 && gstore) ? 0 : kBoxes); bx += NW) {
            // NW boxes' accumulator columns per TMEM wait (512-column tiles:
            // two), each box through its own staging buffer
            uint32_t r[NW][32];
            if (NW == 1) {
                // the previous store from this buffer has finished reading it
                if (lane == 0) ptx::bulk_wait_read<0>();
                __syncwarp();
            }
#pragma unroll
            for (int j = 0; j < NW; ++j) ptx::tmem_ld_32x32b_x32(taddr + (bx + j) * kEpiBoxCols, r[j]);
            ptx::tmem_ld_wait();
            if (bx + NW == kBoxes) {
                // this warp's reads of the accumulator are done: one arrival per warp
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (PAIR == 1) ptx::mbar_arrive(&s.tempty[acc]);
                    else ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_u32(&s.tempty[acc]), 0));
                }
            }
#pragma unroll
            for (int j = 0; j < NW; ++j) {
                const uint32_t jb = static_cast<uint32_t>(j) * kEpiBufBytes;
                if (NW > 1) {
                    // the store that last read buffer j (NW boxes ago) has finished reading it
                    if (lane == 0) ptx::bulk_wait_read<NW - 1>();
                    __syncwarp();
                }
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const uint32_t chunk = static_cast<uint32_t>(v) ^ swz;
                    ptx::st_shared_v4(row_addr + jb + chunk * 16,
                                      ptx::pack_bf16x2(__uint_as_float(r[j][8 * v + 0]), __uint_as_float(r[j][8 * v + 1])),
                                      ptx::pack_bf16x2(__uint_as_float(r[j][8 * v + 2]), __uint_as_float(r[j][8 * v + 3])),
                                      ptx::pack_bf16x2(__uint_as_float(r[j][8 * v + 4]), __uint_as_float(r[j][8 * v + 5])),
                                      ptx::pack_bf16x2(__uint_as_float(r[j][8 * v + 6]), __uint_as_float(r[j][8 * v + 7])));
                }
                // the box's generic-proxy writes are visible to the tensor store
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    ptx::tma_store_2d_hint(&p.tmap_out, buf + jb,
                                           nb * kCols + half * (kCols / 2) + (bx + j) * kEpiBoxCols, arow + q * 32,
                                           pol_out);
                    ptx::bulk_commit();
                }
            }
        }
        if (p.mode == kModeReduceScatter) {
            // Publish the partial tile ("cross-GPU sync protocols on PCIe",
            // section 3): the warp's stores of it come before lane 0's
            // acq_rel arrival on the tile's counter with the warp's share of
            // the 64-unit quota (warp barrier, then the release); the arrival
            // that completes the count is elected and release-stores the
            // sequence into the tile's slot.
            static_assert(kChunkRows % (kEpiWarps * PAIR) == 0, "warp shares must sum to the chunk quota");
            __syncwarp();
            if (lane == 0) arrive_and_publish(p.ctrl, t, kChunkRows / (kEpiWarps * PAIR), p.seq);
            __syncwarp();
        }
        if (p.stats && lane == 0) {
            const long long idx = static_cast<long long>(p.trace_tiles) * p.k_slices + t;
            if (idx < p.ctrl.trace_cap)
                atomicMax(reinterpret_cast<unsigned long long*>(p.ctrl.trace + idx), ptx::globaltimer());
        }
    }
    // every store has written global memory before the CTA retires
    if (lane == 0) ptx::bulk_wait<0>();
    __syncwarp();
}

// Role switch, dynamic schedule (single CTAs or CTA pairs): the same roles as
// above, with tiles taken from the round's ticket counter through a
// shared-memory ring instead of a fixed stride.  They are instantiated only in
// the dynamic-schedule kernels (fused_kernel<PAIR, true>).
namespace dyn {

// Entries of the ring published so far.  A CTA pair shares one schedule:
// the pair's first CTA writes both CTAs' rings, so a pair reads its head at
// cluster scope.
template <int PAIR>
__device__ __forceinline__ int ring_published(const ConsumerSmem<PAIR>& s)
{
    return PAIR == 2 ? ptx::ld_acquire_cluster_smem(s.ring_head) : ptx::ld_acquire_cta_smem(s.ring_head);
}

// Dynamic schedule: wait (bounded) until the scheduler has published ring
// entry k.  Returns false on a pipeline timeout.
template <int PAIR>
__device__ __forceinline__ bool ring_wait(const FusedParams& p, const ConsumerSmem<PAIR>& s, int k)
{
    if (ring_published<PAIR>(s) > k) return true;
    const uint64_t start = ptx::globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (ring_published<PAIR>(s) > k) return true;
        if ((i & 63) == 0 && ptx::globaltimer() - start > static_cast<uint64_t>(p.pipe_timeout_ns)) {
            record_error(p.ctrl, kErrTimeout);
            return false;
        }
        __nanosleep(32);
    }
}

// The k-th tile of this unit (k counts from 0): u + k * n_units statically,
// or ring entry k.  Returns false when the unit has no k-th tile.
template <int PAIR, bool DYN>
__device__ __forceinline__ bool kth_tile(const FusedParams& p, const ConsumerSmem<PAIR>& s, const Schedule<PAIR>& sc,
                                         int k, int& t)
{
    if constexpr (!DYN) {
        t = sc.unit + k * sc.n_units;
        return t < sc.n_tiles;
    }
    if (!ring_wait<PAIR>(p, s, k)) return false;
    t = s.ring[k % kRing];
    return t >= 0;
}

// Dynamic schedule (role switch): the gate warp is also the CTA's scheduler.
// It takes the next tile from the round's ticket counter once the TMA warp
// has issued half of the current tile's loads -- early enough that the new
// tile's gates are passed before the pipeline drains, late enough that no
// CTA holds a tile another could start sooner -- publishes it in
// the ring (CTA-scope release) and then waits for that tile's gates.  A ring
// entry is reused only after the epilogue warps have started its tile.  A
// ticket past the last tile publishes -1 and ends every role.  In a CTA pair
// the first CTA's gate warp schedules for both: it also waits for the other
// CTA's epilogue warps before it reuses an entry, writes the tile into both
// rings and releases both heads at cluster scope; the second CTA's gate
// warp reads its ring like the other roles.
template <int PAIR>
__device__ int sched_next(const FusedParams& p, const ConsumerSmem<PAIR>& s, const Schedule<PAIR>& sc, int k)
{
    const uint32_t lane = ptx::lane_id();
    int t = -1;
    if (PAIR == 2 && sc.rank != 0) {
        if (lane == 0 && ring_wait<PAIR>(p, s, k)) t = s.ring[k % kRing];
        return __shfl_sync(0xffffffffu, t, 0);
    }
    if (lane == 0) {
        bool room = true;
        const int need_epi = k >= kRing ? kEpiWarps * (k - kRing + 1) : 0;
        const uint32_t peer_epi = PAIR == 2 ? ptx::mapa_shared(ptx::smem_u32(s.epi_started), 1) : 0u;
        const uint64_t start = ptx::globaltimer();
        const int need_kb = k * p.n_kb - p.n_kb / 2;
        for (uint32_t i = 1; ptx::ld_acquire_cta_smem(s.tma_done) < need_kb ||
                             ptx::ld_acquire_cta_smem(s.epi_started) < need_epi ||
                             (PAIR == 2 && ptx::ld_acquire_cluster_remote(peer_epi) < need_epi); ++i) {
            if ((i & 63) == 0 && ptx::globaltimer() - start > static_cast<uint64_t>(p.pipe_timeout_ns)) {
                record_error(p.ctrl, kErrTimeout);
                room = false;
                break;
            }
            __nanosleep(32);
        }
        if (room) {
            t = ptx::atom_add_relaxed_gpu(p.ctrl.work, 1);
            if (t >= sc.n_tiles) t = -1;
        }
        if (PAIR == 2) {
            for (uint32_t r = 0; r < 2; ++r) {
                ptx::st_cluster_remote(ptx::mapa_shared(ptx::smem_u32(&s.ring[k % kRing]), r), t);
                ptx::st_release_cluster_remote(ptx::mapa_shared(ptx::smem_u32(s.ring_head), r), k + 1);
            }
        } else {
            s.ring[k % kRing] = t;
            ptx::st_release_cta_smem(s.ring_head, k + 1);
        }
    }
    return __shfl_sync(0xffffffffu, t, 0);
}

template <int PAIR, bool DYN>
__device__ void consumer_gate(const FusedParams& p, const ConsumerSmem<PAIR>& s, const Schedule<PAIR>& sc)
{
    const uint32_t lane = ptx::lane_id();
    unsigned long long polls = 0;
    int passed = 0;
    for (int k = 0;; ++k) {
        int t;
        if constexpr (DYN) {
            t = sched_next<PAIR>(p, s, sc, k);
            if (t < 0) break;
            if (!p.gated) continue;
        } else if (!kth_tile<PAIR, DYN>(p, s, sc, k, t)) {
            break;
        }
        const int mb = sc.row_block(p, t);
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

// Weight (B) cursor of the TMA lane.  B does not depend on the producers, so
// its k-blocks are loaded ahead of the gate: a stage's B boxes are issued (and
// the stage's full barrier armed for A + B bytes) as soon as the stage is
// free, and the stage's A box follows once the slice's gate has passed.
template <int PAIR>
struct BCursor {
    int k;                    // index of the cursor's tile in this unit's schedule
    int t, kb, brow, n0;      // next k-block to load: tile, k-block, B row base, B column base
    bool have;                // t is known (a dynamic schedule publishes tiles as it goes)
    int issued;               // stages armed so far
    uint32_t stage, phase;
    uint64_t pol;             // L2 policy of the weight loads
};

// Resolve the cursor's tile: 1 = known (t >= n_tiles: no more tiles), 0 = not
// published yet (only without `block`), -1 = pipeline timeout.
template <int PAIR, bool DYN>
__device__ __forceinline__ int b_resolve(const FusedParams& p, const ConsumerSmem<PAIR>& s, const Schedule<PAIR>& sc,
                                         BCursor<PAIR>& b, bool block)
{
    if (b.have) return 1;
    int t;
    if constexpr (!DYN) {
        t = sc.unit + b.k * sc.n_units;
    } else {
        if (ring_published<PAIR>(s) <= b.k) {
            if (!block) return 0;
            if (!ring_wait<PAIR>(p, s, b.k)) return -1;
        }
        t = s.ring[b.k % kRing];
        if (t < 0) t = sc.n_tiles;
    }
    b.t = t;
    b.have = true;
    if (t < sc.n_tiles) {
        const int mb = sc.row_block(p, t);
        b.brow = (p.mode == kModeDispatch) ? p.blk_expert[mb] * p.K
               : (p.mode == kModeReduceScatter) ? sc.shard(p, t) * p.K : 0;
        b.n0 = sc.col_block(p, t) * kTileN + static_cast<int>(sc.rank) * (kTileN / PAIR);
    }
    return 1;
}

// Arm the cursor's stage and issue its B boxes (the stage must be free).
template <int PAIR, bool DYN>
__device__ __forceinline__ void b_issue(const FusedParams& p, const ConsumerSmem<PAIR>& s, const Schedule<PAIR>& sc,
                                        BCursor<PAIR>& b)
{
    using T = Tile<PAIR>;
    uint8_t* bdst = s.b + b.stage * T::kStageB;
    // one 3-D load per kWBlocks 64-column blocks (measured: each tensor-load
    // instruction stalls the MMA stream, two 2-D boxes per k-block cost 9.5
    // clocks per pair MMA more than one 3-D box)
    static_assert(T::kBBoxes % kWBlocks == 0, "whole weight loads per stage");
    if (PAIR == 1) {
        ptx::mbar_arrive_expect_tx(&s.full[b.stage], T::kStageBytes);
#pragma unroll
        for (int j = 0; j < T::kBBoxes; j += kWBlocks)
            ptx::tma_load_3d_hint(bdst + j * (kTileK * 128), &p.tmap_b, &s.full[b.stage], 0, b.brow + b.kb * kTileK,
                                  b.n0 / 64 + j, b.pol);
    } else {
        // both CTAs' bytes are counted on the first CTA's barrier
        if (sc.rank == 0) ptx::mbar_arrive_expect_tx(&s.full[b.stage], PAIR * T::kStageBytes);
        const uint32_t bar0 = ptx::mapa_shared(ptx::smem_u32(&s.full[b.stage]), 0);
#pragma unroll
        for (int j = 0; j < T::kBBoxes; j += kWBlocks)
            ptx::tma_load_3d_pair_hint(bdst + j * (kTileK * 128), &p.tmap_b, bar0, 0, b.brow + b.kb * kTileK,
                                       b.n0 / 64 + j, b.pol);
    }
    ++b.issued;
    if (++b.stage == T::kStages) {
        b.stage = 0;
        b.phase ^= 1u;
    }
    if (++b.kb == p.n_kb) {
        b.kb = 0;
        ++b.k;
        b.have = false;
        // a fixed schedule knows the next tile: resolve it at once
        if constexpr (!DYN) b_resolve<PAIR, DYN>(p, s, sc, b, false);
    }
}

// Arm stages until the cursor has armed `upto` stages (blocking on free
// stages and unpublished tiles only when `block`).  Returns false on a
// pipeline timeout.
template <int PAIR, bool DYN>
__device__ __forceinline__ bool b_run(const FusedParams& p, const ConsumerSmem<PAIR>& s, const Schedule<PAIR>& sc,
                                      BCursor<PAIR>& b, int upto, bool block)
{
    while (b.issued < upto) {
        const int r = b_resolve<PAIR, DYN>(p, s, sc, b, block);
        if (r < 0) return false;
        if (r == 0 || b.t >= sc.n_tiles) return true;
        if (block) {
            if (!mbar_wait(&s.empty[b.stage], b.phase ^ 1u, p.ctrl, p.pipe_timeout_ns)) return false;
        } else if (!ptx::mbar_try_wait(&s.empty[b.stage], b.phase ^ 1u)) {
            return true;
        }
        b_issue<PAIR, DYN>(p, s, sc, b);
    }
    return true;
}

// TMA lane: wait until the gate warp has passed gate number `idx` (bounded),
// arming free stages with B meanwhile.
template <int PAIR, bool DYN>
__device__ __forceinline__ bool wait_gate(const FusedParams& p, const ConsumerSmem<PAIR>& s, const Schedule<PAIR>& sc,
                                          BCursor<PAIR>& b, int a_count, int idx)
{
    using T = Tile<PAIR>;
    if (ptx::ld_acquire_cta_smem(s.gates_passed) > idx) return true;
    const uint64_t start = ptx::globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (!b_run<PAIR, DYN>(p, s, sc, b, a_count + T::kStages, false)) return false;
        if (ptx::ld_acquire_cta_smem(s.gates_passed) > idx) return true;
        if ((i & 63) == 0 && ptx::globaltimer() - start > static_cast<uint64_t>(p.pipe_timeout_ns)) {
            record_error(p.ctrl, kErrTimeout);
            return false;
        }
        __nanosleep(20);
    }
}

// TMA warp: per tile and K-slice, wait for the slice's gate, then stream the
// slice's A k-blocks into stages whose B the cursor above has already
// loaded.  One lane issues everything.
template <int PAIR, bool DYN>
__device__ void consumer_tma(const FusedParams& p, const ConsumerSmem<PAIR>& s, const Schedule<PAIR>& sc)
{
    using T = Tile<PAIR>;
    if (ptx::lane_id() != 0) return;
    BCursor<PAIR> b;
    b.k = 0;
    b.t = 0;
    b.kb = 0;
    b.have = false;
    b.issued = 0;
    b.stage = 0;
    b.phase = 0;
    b.pol = stream_policy(p, kHintBLast, 0);
    const uint64_t pol_a = stream_policy(p, 0, kHintAFirst);
    uint32_t stage = 0;
    int a_count = 0;
    int gate_idx = 0;
    for (int k = 0;; ++k) {
        int t;
        if (!kth_tile<PAIR, DYN>(p, s, sc, k, t)) break;
        const int arow = sc.a_row(p, t);
        for (int sl = 0; sl < p.k_slices; ++sl, ++gate_idx) {
            if (p.gated) {
                if (!wait_gate<PAIR, DYN>(p, s, sc, b, a_count, gate_idx)) return;
                // the rows were written through the generic proxy; order them
                // before this thread's tensor-memory-access (async proxy) reads
                ptx::fence_proxy_async_global();
            }
            const int kb1 = kb_begin(p, sl + 1);
            for (int kb = kb_begin(p, sl); kb < kb1; ++kb) {
                // this k-block's stage is armed and holds (or receives) its B
                if (!b_run<PAIR, DYN>(p, s, sc, b, a_count + 1, true)) return;
                uint8_t* adst = s.a + stage * T::kStageA;
                if (PAIR == 1) {
                    ptx::tma_load_2d_hint(adst, &p.tmap_a, &s.full[stage], kb * kTileK, arow, pol_a);
                } else {
                    const uint32_t bar0 = ptx::mapa_shared(ptx::smem_u32(&s.full[stage]), 0);
                    ptx::tma_load_2d_pair_hint(adst, &p.tmap_a, bar0, kb * kTileK, arow, pol_a);
                }
                ++a_count;
                if (++stage == T::kStages) stage = 0;
            }
            if constexpr (DYN) ptx::st_release_cta_smem(s.tma_done, k * p.n_kb + kb1);
        }
    }
}

// MMA warp: one lane (of the pair's first CTA) issues the MMAs.
template <int PAIR, bool DYN>
__device__ void consumer_mma(const FusedParams& p, const ConsumerSmem<PAIR>& s, const Schedule<PAIR>& sc,
                             uint32_t tmem_base)
{
    using T = Tile<PAIR>;
    if (ptx::lane_id() != 0 || sc.rank != 0) return;
    uint32_t stage = 0, phase = 0;
    for (int local = 0;; ++local) {
        int t;
        if (!kth_tile<PAIR, DYN>(p, s, sc, local, t)) break;
        const uint32_t acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!mbar_wait(&s.tempty[acc], acc_phase ^ 1u, p.ctrl, p.pipe_timeout_ns)) return;
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + acc * kTileN;
        for (int kb = 0; kb < p.n_kb; ++kb) {
            // the stage's TMA bytes have landed (the barrier's transaction
            // count); the MMAs below read them through the async proxy and
            // are issued after this wait in program order.  No tcgen05
            // thread-sync fence here: measured, it costs 14 clocks per MMA
            // (142.5 instead of 128) once the stages rotate
            if (!mbar_wait(&s.full[stage], phase, p.ctrl, p.pipe_timeout_ns)) return;
            const uint32_t a0 = ptx::smem_u32(s.a + stage * T::kStageA);
            const uint32_t b0 = ptx::smem_u32(s.b + stage * T::kStageB);
#pragma unroll
            for (int k = 0; k < kTileK / kUmmaK; ++k) {
                // A: K-major, 128B swizzle; +32 B per 16-element k step inside
                //    the swizzle row; 8-row groups 1024 B apart.
                const uint64_t ad = ptx::smem_desc_sw128(a0 + k * 32, 16, 1024);
                // B: MN-major, 128B swizzle; +2048 B per 16 k-rows; 8-k-row
                //    groups 1024 B apart; 64-column blocks 8 KB apart.
                const uint64_t bd = ptx::smem_desc_sw128(b0 + k * 2048, kTileK * 128, 1024);
                if (PAIR == 1) ptx::umma_bf16(d, ad, bd, T::kIdesc, (kb | k) != 0);
                else ptx::umma_bf16_pair(d, ad, bd, T::kIdesc, (kb | k) != 0);
            }
            if (PAIR == 1) ptx::umma_commit(&s.empty[stage]);
            else ptx::umma_commit_pair(&s.empty[stage], 0x3);
            if (++stage == T::kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (PAIR == 1) ptx::umma_commit(&s.tfull[acc]);
        else ptx::umma_commit_pair(&s.tfull[acc], 0x3);
    }
}

// Epilogue warps: TMEM -> registers -> bf16 (round to nearest even) ->
// shared memory -> TMA tensor store.  Warp w reads TMEM lane quarter w % 4
// (the quarter its position allows), i.e. 32 output rows, and one half of
// the 256 accumulator columns, as four 32 x 32 boxes.  A box is written into
// the warp's 2 KB buffer in the 64-byte swizzled layout the store's tensor
// map expects (16-byte chunk j of 64-byte row r at chunk j ^ ((r / 2) % 4):
// the eight rows a quarter-warp writes hit distinct banks), then one lane
// stores it; rows past the output's extent (the ragged tail of M) are
// clipped by the store.  The accumulator is released as soon as its last
// columns are in registers.
template <int PAIR, bool DYN>
__device__ void consumer_epilogue(const FusedParams& p, const ConsumerSmem<PAIR>& s, const Schedule<PAIR>& sc,
                                  uint32_t tmem_base)
{
    const int warp = threadIdx.x / 32;
    const uint32_t lane = ptx::lane_id();
    const int q = warp & 3;
    const int half = (warp - kEpiWarp0) / 4;
    const uint8_t* buf = s.epi + (warp - kEpiWarp0) * kEpiBufBytes;
    const uint32_t row_addr = ptx::smem_u32(buf) + lane * (kEpiBoxCols * 2);
    const uint32_t swz = (lane >> 1) & 3u;
    const uint64_t pol_out = stream_policy(p, 0, kHintOutFirst);
    for (int local = 0;; ++local) {
        int t;
        if (!__all_sync(0xffffffffu, kth_tile<PAIR, DYN>(p, s, sc, local, t))) break;
        // the ring entry is read: the scheduler may reuse it kRing tiles on
        if (DYN && lane == 0) {
            if (PAIR == 2) ptx::red_add_release_cluster_smem(s.epi_started, 1);   // the first CTA schedules
            else ptx::red_add_release_cta_smem(s.epi_started, 1);
        }
        const int arow = sc.a_row(p, t);
        const int nb = sc.col_block(p, t);
        const uint32_t acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        const bool arrived = mbar_wait(&s.tfull[acc], acc_phase, p.ctrl, p.pipe_timeout_ns);
        if (!__all_sync(0xffffffffu, arrived)) break;
        ptx::tc_fence_after();
        if (p.stats && lane == 0) {
            const long long idx = static_cast<long long>(p.trace_tiles) * (p.k_slices + 1) + t;
            if (idx < p.ctrl.trace_cap)
                atomicMax(reinterpret_cast<unsigned long long*>(p.ctrl.trace + idx), ptx::globaltimer());
        }
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kTileN + half * (kTileN / 2);
#pragma unroll 1
        for (int bx = 0; bx < kTileN / 2 / kEpiBoxCols; ++bx) {
            // the previous store from this buffer has finished reading it
            if (lane == 0) ptx::bulk_wait_read<0>();
            __syncwarp();
            {
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(taddr + bx * kEpiBoxCols, r);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const uint32_t chunk = static_cast<uint32_t>(v) ^ swz;
                    ptx::st_shared_v4(row_addr + chunk * 16,
                                      ptx::pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1])),
                                      ptx::pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3])),
                                      ptx::pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5])),
                                      ptx::pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7])));
                }
            }
            if (bx == kTileN / 2 / kEpiBoxCols - 1) {
                // this warp's reads of the accumulator are done: one arrival per warp
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (PAIR == 1) ptx::mbar_arrive(&s.tempty[acc]);
                    else ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_u32(&s.tempty[acc]), 0));
                }
            }
            // the box's generic-proxy writes are visible to the tensor store
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                ptx::tma_store_2d_hint(&p.tmap_out, buf, nb * kTileN + half * (kTileN / 2) + bx * kEpiBoxCols,
                                       arow + q * 32, pol_out);
                ptx::bulk_commit();
            }
        }
        if (p.mode == kModeReduceScatter) {
            // Publish the partial tile ("cross-GPU sync protocols on PCIe",
            // section 3): once this warp's stores have written global memory,
            // it arrives on the tile's counter with its share of the
            // 64-unit quota; the arrival that completes the count is elected
            // and release-stores the sequence into the tile's slot.
            if (lane == 0) {
                ptx::bulk_wait<0>();
                ptx::fence_proxy_async_global();
            }
            __syncwarp();
            static_assert(kChunkRows % (kEpiWarps * PAIR) == 0, "warp shares must sum to the chunk quota");
            if (lane == 0) arrive_and_publish(p.ctrl, t, kChunkRows / (kEpiWarps * PAIR), p.seq);
            __syncwarp();
        }
        if (p.stats && lane == 0) {
            const long long idx = static_cast<long long>(p.trace_tiles) * p.k_slices + t;
            if (idx < p.ctrl.trace_cap)
                atomicMax(reinterpret_cast<unsigned long long*>(p.ctrl.trace + idx), ptx::globaltimer());
        }
    }
    // every store has written global memory before the CTA retires
    if (lane == 0) ptx::bulk_wait<0>();
    __syncwarp();
}

}  // namespace dyn

// Embedded producers: in a launch without producer CTAs, the consumer CTAs'
// warps between the gate warp and the stage waiter (4 per CTA) copy the
// rows, with the producers' item order, counters and seeds (producer.cuh),
// dealt across every CTA.
// They own no mbarrier, TMEM column or ring entry, so they skip the
// prologue: they count toward its barrier without waiting for it and start
// as soon as the previous kernel's output (the plan) is visible.
constexpr int kFirstCopyWarp = kGateWarp + 1;

template <int PAIR>
__device__ __forceinline__ void embedded_producer(const FusedParams& p)
{
    constexpr int kCopyWarps = kWaitWarp - kFirstCopyWarp;
    const int warp = threadIdx.x / 32;
    if (PAIR == 2) ptx::cluster_arrive_relaxed();
    ptx::grid_dep_wait();
    const int gw = (warp - kFirstCopyWarp) * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x);
    const int n_gw = kCopyWarps * static_cast<int>(gridDim.x);
    if (warp == kFirstCopyWarp && ptx::lane_id() == 0) stat_min(p, kStatProdStartNs, ptx::globaltimer());
    seed_counters(p, gw, n_gw, true);
    if (p.item_rows <= 16) copy_items<1>(p, gw, n_gw);
    else if (p.item_rows == 32) copy_items<2>(p, gw, n_gw);
    else copy_items<4>(p, gw, n_gw);
    seed_counters(p, gw, n_gw, false);
    __syncwarp();
    if (ptx::lane_id() == 0) stat_max(p, kStatProdEndNs, ptx::globaltimer());
    // the prologue's cluster barrier completes before the teardown's
    if (PAIR == 2) ptx::cluster_wait();
}

template <int PAIR, bool DYN, bool EMB, int NW = 1>
__device__ void consumer(const FusedParams& p, uint8_t* smem, int cid)
{
    constexpr int ST = NW == 2 ? kWideStages : (EMB ? emb_stages_for(PAIR) : stages_for(PAIR));
    using T = Tile<PAIR, ST, NW>;
    const int warp = threadIdx.x / 32;
    const ConsumerSmem<PAIR> s = consumer_smem<PAIR, ST, NW>(smem);
    if (EMB && warp >= kFirstCopyWarp && warp < kWaitWarp) {
        embedded_producer<PAIR>(p);
        // the teardown barrier: TMEM is freed after every warp is done
        if (PAIR == 1) ptx::bar_sync_unaligned(0, kThreads);
        else ptx::cluster_sync();
        return;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < T::kStages; ++i) {
            ptx::mbar_init(&s.full[i], 1);
            ptx::mbar_init(&s.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&s.tfull[i], 1);
            ptx::mbar_init(&s.tempty[i], kEpiWarps * PAIR);
        }
        *s.gates_passed = 0;
        *s.ring_head = 0;
        *s.epi_started = 0;
        *s.tma_done = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&p.tmap_a);
        ptx::prefetch_tmap(&p.tmap_b);
        ptx::prefetch_tmap(&p.tmap_out);
        stat_min(p, kStatConsStartNs, ptx::globaltimer());
    }
    if (warp == 1) {
        if (PAIR == 1) {
            ptx::tmem_alloc(s.tmem_slot, kTmemCols);
            ptx::tmem_relinquish();
        } else {
            ptx::tmem_alloc_pair(s.tmem_slot, kTmemCols);
            ptx::tmem_relinquish_pair();
        }
    }
    ptx::tc_fence_before();
    // barriers initialised and TMEM allocated in both CTAs before any
    // cross-CTA arrival or load (copy warps only arrive)
    if (PAIR == 2) ptx::cluster_sync();
    else if (EMB) ptx::bar_sync_unaligned(1, (kFirstCopyWarp + 1) * 32);   // warps 0-10 and the waiter
    else __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *s.tmem_slot;
    // the prologue above overlaps the previous kernel; the schedule (a
    // dispatch plan's block count), the gates and the operands are its output
    ptx::grid_dep_wait();
    const Schedule<PAIR> sc = make_schedule<PAIR>(p, cid);

    if constexpr (DYN) {
        // role switch: tiles from the ticket counter
        if (warp == 0) dyn::consumer_tma<PAIR, true>(p, s, sc);
        else if (warp == 1) dyn::consumer_mma<PAIR, true>(p, s, sc, tmem_base);
        else if (warp < kEpiWarp0 + kEpiWarps) dyn::consumer_epilogue<PAIR, true>(p, s, sc, tmem_base);
        else if (warp == kGateWarp) dyn::consumer_gate<PAIR, true>(p, s, sc);
    } else {
        if (warp == 0) consumer_tma<PAIR, ST, NW>(p, s, sc);
        else if (warp == 1) consumer_mma<PAIR, ST, NW>(p, s, sc, tmem_base);
        else if (warp < kEpiWarp0 + kEpiWarps) consumer_epilogue<PAIR, NW>(p, s, sc, tmem_base);
        else if (warp == kWaitWarp) consumer_stage_waiter<PAIR, ST>(p, s, sc);
        else if (warp == kGateWarp && p.gated) consumer_gate<PAIR>(p, s, sc);
        else if (warp >= kGateWarp && p.mode == kModeReduceScatter && p.rs_epi) {
            // no producer CTAs: the gate warp and the spare warps add the
            // per-round quota seeds of the counters this round does not fill,
            // then sum the output tiles this CTA (pair) owns
            constexpr int kSpare = kWaitWarp - kGateWarp;
            seed_counters(p, (warp - kGateWarp) * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x),
                          kSpare * static_cast<int>(gridDim.x), false);
            rs_reduce_owned(p, sc.unit, sc.n_units, static_cast<int>(sc.rank), kGateWarp);
        }
    }
    __syncwarp();

    // teardown: every role of both CTAs has finished before TMEM is freed
    // (and before a CTA whose shared memory the peer reads exits)
    ptx::tc_fence_before();
    if (PAIR == 2) ptx::cluster_sync();
    else if (EMB) ptx::bar_sync_unaligned(0, kThreads);
    else __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        if (PAIR == 1) ptx::tmem_dealloc(tmem_base, kTmemCols);
        else ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
    }
    if (threadIdx.x == 0) stat_max(p, kStatConsEndNs, ptx::globaltimer());
    // role switch: with its tiles done, every warp of the CTA takes
    // reduction items from the round's ticket counter
    if (p.mode == kModeReduceScatter && p.rs_join) rs_reduce(p);
}

}  // namespace tovl
