// ctrl.cuh -- control-plane layout, kernel parameter blocks and constants.
//
// The control plane (slots, counters, status) lives in its own allocation,
// apart from the data plane, as the NVLink-atomics page recommends (section
// 3.1: synchronisation metadata kept separate from data).  Every counter is
// monotonic and never reset ("cross-GPU sync protocols on PCIe", section 2):
// after the R-th call on a handle every slot holds R, every chunk counter
// 64*R and every row-block counter 128*R.
#pragma once
#include <cstdint>
#include <cuda.h>

namespace tovl {

constexpr int kChunkRows = 64;     // watermark granularity (section 4 of the sync-protocol page)
constexpr int kBlockRows = 128;    // row-block gate = GEMM M tile (section 5)
constexpr int kTileM = 128;
constexpr int kTileN = 256;
constexpr int kTileK = 64;         // 64 bf16 = one 128-byte swizzle row
constexpr int kWBlocks = 2;        // 64-column weight blocks per tensor load (one instruction)
constexpr int kUmmaK = 16;
constexpr int kStages = 4;
constexpr int kThreads = 512;      // 16 warps: TMA, MMA, 8 x epilogue, gate, 4 spare, stage waiter (consumers) / 16 copy warps (producers)
constexpr int kEpiWarp0 = 2;       // first epilogue warp
constexpr int kEpiWarps = 8;       // two per TMEM lane quarter, each owning 128 of the 256 columns
constexpr int kGateWarp = 10;      // polls the protocol ahead of the TMA warp
constexpr int kWaitWarp = 15;      // observes the stages' full barriers for the MMA warp (fixed schedule)
constexpr int kStageBar0 = 2;      // named barrier kStageBar0 + stage: stage hand-off, waiter warp -> MMA warp
constexpr int kStageBarThreads = 64;
constexpr int kTraceCap = 1 << 20; // timeline entries kept when statistics are on
constexpr int kMaxSlices = 8;      // K-slices per chunk watermark
constexpr int kItemInt4 = 512;     // one producer item moves at most 8 KB per pass (16 x 16 B per lane)
constexpr int kItemBytes = kItemInt4 * 16;
constexpr int kMaxShards = 64;
constexpr int kMaxK = 32768;       // a producer ring stage must hold one 64 KB row
constexpr int kMaxExperts = 512;

constexpr int kStageA = kTileM * kTileK * 2;      // 16 KB
constexpr int kStageB = kTileK * kTileN * 2;      // 32 KB
constexpr int kStageBytes = kStageA + kStageB;    // 48 KB
constexpr int kTmemCols = 512;                    // two 128x256 fp32 accumulators
// dynamic shared memory: stages + barriers + 1 KB alignment slack
constexpr int kEpiBoxCols = 32;                   // output box of one epilogue store: 32 rows x 32 columns
constexpr int kEpiBufBytes = 32 * kEpiBoxCols * 2; // 2 KB staging buffer per epilogue warp (64B swizzle)
constexpr int kPairStages = 5;                     // pipeline stages of a CTA-pair consumer (32 KB each)

// Pipeline stages and dynamic shared memory of the fused kernel per consumer
// shape.  Producer CTAs share the launch's shared-memory size, and a producer
// SM's L1 is what is left of the 256 KB: every kilobyte given to shared
// memory is one its loads cannot have in flight, so the stages are as few as
// keep the tensor pipe fed.
constexpr int stages_for(int pair) { return pair == 1 ? kStages : kPairStages; }
// (512-column tiles, nw = 2, give each epilogue warp two staging buffers)
constexpr int smem_for(int pair, int stages, int nw = 1)
{
    return stages * (kStageA + kStageB * nw / pair) + kEpiWarps * kEpiBufBytes * nw + 1024 + 1024;
}
constexpr int smem_bytes(int pair) { return smem_for(pair, stages_for(pair)); }
// Launches without producer CTAs (embedded producers) leave no SM's L1 to
// protect: CTA pairs take a sixth stage there (measured: the uniform and Zipf
// dispatch rounds 2.5-3 % faster; with producer CTAs it cost the TP call 2 us).
constexpr int kEmbPairStages = 6;
constexpr int emb_stages_for(int pair) { return pair == 2 ? kEmbPairStages : stages_for(pair); }
constexpr int smem_bytes_emb(int pair) { return smem_for(pair, emb_stages_for(pair)); }
// 256 x 512 CTA-pair tiles (dispatch with embedded producers): each CTA
// stages A 16 KB + 256 weight columns 32 KB per k-block, four stages.
constexpr int kWideStages = 4;
constexpr int smem_bytes_wide() { return smem_for(2, kWideStages, 2); }

// Device status codes (mirror tovl.h).
enum : int {
    kOk = 0,
    kErrInvalid = 1,
    kErrUnsupported = 2,
    kErrCuda = 3,
    kErrTimeout = 4,
    kErrOom = 5,
};

// Statistics slots (64-bit), only written when stats are enabled.
enum : int {
    kStatGatePolls = 0,      // acquire polls issued by consumer gates
    kStatConsStartNs = 1,    // earliest consumer start (%globaltimer)
    kStatConsEndNs = 2,      // latest consumer end
    kStatProdStartNs = 3,    // earliest producer start
    kStatProdEndNs = 4,      // latest producer end (all rows published)
    kStatTimeouts = 5,
    kNumStats = 8,
};

struct Ctrl {
    int* slot;            // [n_chunk_cap]  chunk watermark slots (single writer per round)
    int* cnt;             // [n_chunk_cap]  chunk arrival counters
    int* rbcnt;           // [n_block_cap]  row-block arrival counters
    int* status;          // [1] sticky error code
    int* abort_seq;       // [1] highest sequence that gave up waiting
    int* work;            // [1] item tickets of a round whose items are shared out dynamically (zeroed per round)
    unsigned long long* stats;   // [kNumStats]
    long long* pub_ns;    // [n_chunk_cap * n_slices]  publish time of each chunk slice (stats / stamps)
    long long* obs_ns;    // [n_chunk_cap]  first observation time by a waiter (copy sweep)
    long long* trace;     // [trace_cap]  fused kernel timeline: gate-pass times per tile slice, then tile end times
    int trace_cap;
    int n_chunk_cap;
    int n_block_cap;
    int n_slices;         // K-slices per chunk / block; slot, cnt and rbcnt hold n_slices entries per chunk / block
};

// Routing plan produced on the device for one dispatch round.
struct Plan {
    int* counts;          // [E]
    int* off;             // [E+1] padded segment starts (internal copy)
    int* prev_off;        // [E+1] previous round's layout (zero-padding decision)
    int* seg_count;       // [n_seg][E] per-segment counts, then segment prefixes
    int* local_rank;      // [T*k] rank of each pair inside its segment and expert
    int* dst;             // [T*k] destination row of each pair
    int* src_of_dst;      // [row cap] token of each destination row, -1 = padding
    int* pad;             // [block cap] padding rows per block (counter seed)
    int* blk_expert;      // [block cap]
    int* meta;            // [4] m_pad, n_blocks, zero_padding, error
    // CTA-pair row tiles over 128-row segments: [0] = their count, then per
    // tile 2 * (first block) + 1 if the next block is in the same segment
    // (else the pair's second CTA computes a phantom half that is never
    // stored); null when not wanted
    int* pair_tab;        // [1 + block cap]
};

enum : int { kModeGather = 0, kModeDispatch = 1, kModeReduceScatter = 2 };

// L2 eviction priorities per stream of a fused call (FusedParams::l2_hints):
// producer source loads evict-last (a dispatch reads a token row k times) or
// evict-first (read once), producer destination stores evict-last (the GEMM
// reads them later), A tensor loads evict-first, weight (B) tensor loads
// evict-last, output tensor stores evict-first (never read in the call).
enum : int {
    kHintSrcLast = 1,
    kHintOutFirst = 2,
    kHintAFirst = 4,
    kHintBLast = 8,
    kHintDstLast = 16,
    kHintSrcFirst = 32,
};

struct FusedParams {
    CUtensorMap tmap_a;   // A: gathered / dispatched rows [rows][K] bf16, box 64 x 128, 128B swizzle
    CUtensorMap tmap_b;   // B: weights [(E*)K][N] bf16 row-major (MN-major operand) viewed as
                          // [N/64][(E*)K][64], box 64 x 64 x kWBlocks (kWBlocks 64-column blocks per load)
    CUtensorMap tmap_out; // out [rows][N] bf16, box 32 x 32, 64B swizzle (rows past the extent are not stored)
    int mode;
    int M;                // gather: rows of the gathered buffer
    int N, K;
    int n_kb;             // K / 64
    int n_nb;             // N / 256
    int n_producers;
    int n_consumers;
    int gated;            // consumers wait on the protocol before loading A
    int seq;
    int gate_seq;         // sequence the consumer gates wait for (seq, unless a fault is injected)
    long long timeout_ns; // bound of a gate wait on other CTAs
    long long pipe_timeout_ns;  // bound of a wait on this CTA's own pipeline (outlasts a gate timeout)
    int stats;
    int row_bytes;        // K * 2
    int k_slices;         // K-slices in use this call (<= ctrl.n_slices); slices beyond are seeded
    int wave_blocks;      // row blocks the consumers' first wave covers (producer ordering group)
    int item_rows;        // rows per producer item (a power of two dividing 64)
    int producer_mode;    // 0: vector copies through registers; 1: bulk loads staged in shared memory
    int trace_tiles;      // tile count bound that lays out the timeline (gate times, then end times)
    int l2_hints;         // L2 eviction priorities of the call's streams (kHint* bits)
    // gather sources
    const void* shard[kMaxShards];
    int n_shards;
    int rows_per_shard;
    // dispatch sources
    const void* x;
    const int* src_of_dst;
    const int* pad;
    const int* pair_tab;  // Plan::pair_tab when CTA pairs run 128-row dispatch segments, else null
    const int* blk_expert;
    const int* meta;
    // combine sources (gather mode with a row table)
    const int* src_rows;  // non-null: destination row r copies row src_rows[r] of x
    const int* rows_valid;  // non-null: the round has rows only if rows_valid[1] > 0 (plan block count)
    const float* gate_w;  // [T*k] combine weights
    void* combined;       // [T][N] bf16 combined rows
    int n_reducers;
    int T, k;
    // reduce-scatter: consumers write shard partials (out, [S][M][N]) and
    // publish each partial tile; producers sum the S partials into rs_out
    int rs_tiles;         // partial tiles: S x output tiles; tile t publishes counter t
    int rs_pair;          // rows of an output tile / 128
    int rs_join;          // consumers take reduction items once their tiles are done (role switch)
    int rs_epi;           // no producer CTAs: output tile o is summed in the epilogue of the CTA (pair)
                          // that computes shard (o mod S)'s partial of it
    int dyn;              // consumer tiles handed out by a ticket counter (ctrl.work, zeroed by the plan kernel)
    int join;             // producer CTAs become consumers once their copies are done (role switch)
    int embedded;         // no producer CTAs: the consumer CTAs' spare warps copy the rows
    int wide;             // CTA pairs compute 256 x 512 tiles (n_nb counts 512-column blocks; embedded dispatch)
    void* rs_out;         // [M][N] bf16
    // destinations
    void* gathered;       // gathered / dispatched buffer
    void* out;            // [rows][N] bf16
    int out_rows;         // gather: M; dispatch: row capacity of out
    Ctrl ctrl;
};

struct PlanParams {
    const int* topk;      // [T*k]
    int n_pairs;          // T*k
    int k;
    int E;
    int n_seg;
    int row_cap;          // rows available in the dispatched buffer
    int block_cap;        // row-block counters available
    int force_zero;       // host: buffer changed, re-zero padding rows
    int* expert_offsets;  // caller-visible [E+1]
    Plan plan;
    int* status;
    int* work;            // ticket counter of the fused kernel that follows (zeroed here)
    int align;            // expert segments start at multiples of this many rows (128 or 256)
};

struct CopyParams {
    const uint8_t* src;
    uint8_t* dst;
    const int* perm;      // dst row of each src row
    long long n_rows;
    int row_bytes;
    int n_chunks;         // chunks touched by this copy
    int gated;
    int n_copiers;        // CTAs that copy; the remaining CTAs wait on slots
    int seq;
    long long timeout_ns;
    long long pipe_timeout_ns;
    int copy_mode;
    int stamps;           // record publish / observe times
    Ctrl ctrl;
};

}  // namespace tovl
