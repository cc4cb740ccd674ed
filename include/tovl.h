/*
 * tovl.h -- C ABI of the tovl library: token-row movement fused with a bf16
 * tensor-core GEMM on one NVIDIA GB300 (sm_103a).
 *
 * The method: producer CTAs move token rows into one gathered buffer while
 * consumer CTAs run a GEMM that starts on each 128-row block as soon as its
 * rows are complete.  Completion follows the single-writer slot protocol of
 * the Astro Bear page "Fused compute/communication operators (4): cross-GPU
 * sync protocols on PCIe -- single writer, election and watermarks":
 *   section 2  slots hold monotonically increasing sequence numbers that are
 *              never reset; round k waits for a value >= k;
 *   section 3  many writers are counted with a local acq_rel atomic and the
 *              last arrival is elected to publish with a release store;
 *   section 4  one watermark slot per 64-row chunk;
 *   section 5  row-block counters take release reductions and are pre-seeded
 *              with the padding count, so real arrivals reach 128 exactly.
 * The "ranks" of the pages are logical shards held in this GPU's memory; the
 * library uses no peer memory and no collectives.
 *
 * Conventions for every entry point:
 *   - Pointers named as device pointers must point to device memory of the
 *     handle's GPU, 16-byte aligned; host pointers are ordinary host memory.
 *   - bf16 tensors are row-major with unit stride in the last dimension.
 *   - The caller owns every buffer and stream; the handle owns only its
 *     control plane (counters, slots, status word, plan scratch) and its
 *     sequence number.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous; one call is one protocol round.  Calls on one handle must
 *     be issued from one host thread, in order, on one stream.
 *   - Return value: TOVL_OK, or an error code from tovl_status.  Argument
 *     errors are detected on the host before anything is enqueued and leave
 *     the handle unchanged.  Errors found on the device (a wait that timed
 *     out, an expert id out of range) are sticky in the handle's status word
 *     and read with tovl_sync_status(); device code never traps.
 *   - There is no CPU fallback: on a machine without a compute-capability
 *     10.3 GPU, tovl_create returns TOVL_ERR_UNSUPPORTED.
 */
#ifndef TOVL_H
#define TOVL_H

#ifdef __cplusplus
extern "C" {
#endif

typedef struct tovl_ctx* tovl_handle;

typedef enum {
    TOVL_OK = 0,
    TOVL_ERR_INVALID = 1,      /* bad argument, shape, alignment or routing */
    TOVL_ERR_UNSUPPORTED = 2,  /* shape or device the kernels do not support */
    TOVL_ERR_CUDA = 3,         /* a CUDA runtime call failed; see tovl_last_error */
    TOVL_ERR_TIMEOUT = 4,      /* a device wait gave up (sticky, from tovl_sync_status) */
    TOVL_ERR_OOM = 5           /* device allocation failed in tovl_create */
} tovl_status;

/* Row-copy mechanism of tovl_gated_copy.  The producers of the fused
 * kernels use 16 warps per CTA; their copy path is option 14. */
typedef enum {
    TOVL_COPY_VECTOR = 0,      /* 16-byte vector loads/stores by warps */
    TOVL_COPY_BULK = 1,        /* bulk asynchronous copies through a shared-memory ring */
    TOVL_COPY_AUTO = 2         /* vector below 8 KB rows, bulk from 8 KB (the default) */
} tovl_copy_mode;

typedef struct {
    int device;                /* CUDA device ordinal */
    int chunk_rows;            /* watermark chunk; must be 64 (or 0 for 64) -- section 4 */
    int gate_rows;             /* GEMM row-block gate; must be 128 (or 0 for 128) -- section 5 */
    int producer_ctas;         /* P; 0 = chosen per call: copy and GEMM time balanced,
                                  then grown while the GEMM keeps its wave count */
    int consumer_ctas;         /* C; 0 = all remaining SMs */
    long long wait_timeout_ns; /* bound of every device wait; 0 = 2 s */
    int copy_mode;             /* tovl_copy_mode of tovl_gated_copy; the default is
                                  TOVL_COPY_AUTO (measured on GB300, gated: 71-91 % of
                                  the HBM copy bandwidth with vector copies from 256 B
                                  to 4 KB rows, 94-96 % with bulk copies at 8-16 KB) */
    long long max_rows;        /* capacity in rows of gathered/dispatched buffers and copies */
    int max_pairs;             /* largest T*k of a dispatch call */
    int max_experts;           /* largest E of a dispatch call (<= 512) */
    int k_slices;              /* 1..8 (0 = 1): each 64-row chunk watermark (and each
                                  128-row block counter) is split into this many
                                  K-ranges, published separately, so a GEMM tile may
                                  start on the first K-range of its rows; 1 = one
                                  watermark per chunk (sections 4-5 exactly) */
} tovl_config;

/* Fills `cfg` with defaults for `device`. */
void tovl_default_config(tovl_config* cfg, int device);

/* Creates a handle: validates `cfg`, checks the device (compute capability
 * 10.3), allocates and zeroes the control plane (chunk slots and counters for
 * max_rows/64 chunks, row-block counters for max_rows/128 blocks, status
 * word, plan scratch).  Sequence number starts at 0.  On failure *out is
 * NULL and nothing stays allocated. */
int tovl_create(tovl_handle* out, const tovl_config* cfg);

/* Frees the handle's device memory after synchronising its last stream.
 * NULL is accepted.  The handle must not be used afterwards. */
int tovl_destroy(tovl_handle h);

/* All-gather of S logical shards followed by a GEMM (the tensor-parallel
 * all-gather + GEMM of the platform page "know your platform", section 3,
 * with the completion protocol of sections 2-5 of the sync page).
 *   shards      host array of S device pointers; shard s is bf16 [R][K]
 *   num_shards  S, 1..64
 *   rows_per_shard R >= 1; M = S*R <= max_rows
 *   K           multiple of 64, at most 32768
 *   W           device, bf16 [K][N]
 *   N           multiple of 256
 *   gathered    device, bf16 [M][K]: receives G[s*R + i] = shard s row i
 *   out         device, bf16 [M][N]: out = G x W, fp32 accumulation,
 *               rounded to nearest even
 * One round: producers copy every row and publish each 64-row chunk; each
 * consumer tile waits for its chunks' slots to reach this round's sequence. */
int tovl_gather_gemm(tovl_handle h, const void* const* shards, int num_shards, int rows_per_shard, int K,
                     const void* W, int N, void* gathered, void* out, void* stream);

/* Rows a dispatch buffer needs: T*k + E*127 rounded up to a multiple of 128. */
long long tovl_dispatch_rows(int T, int k, int E);

/* The same bound for expert segments aligned to `align` rows (128, or 256 with
 * option 17): T*k + E*(align-1) rounded up to a multiple of align; 0 for any
 * other align. */
long long tovl_dispatch_rows_aligned(int T, int k, int E, int align);

/* Dispatch scatter of top-k routed tokens into padded per-expert segments,
 * followed by a grouped GEMM per expert (notify-stage counting of the DeepEP
 * FIFO-pipeline page; row-block counters with padding seeds of section 5).
 *   x           device, bf16 [T][H] (may be null when T = 0)
 *   topk_idx    device, int32 [T][k]: expert of pair (t, j), each in [0, E)
 *               (may be null when T = 0: a round without tokens, whose plan
 *               is empty and whose call still counts as one round)
 *   H           multiple of 64, at most 32768 (the GEMM K)
 *   W           device, bf16 [E][H][N], N multiple of 256
 *   dispatched  device, bf16 [tovl_dispatch_rows(T,k,E)][H]: rows of expert e
 *               occupy [off[e], off[e] + count[e]) in ascending (t, j) order;
 *               the segment is padded with zero rows to a multiple of 128
 *   expert_offsets device, int32 [E+1]: receives off[]; off[E] = padded total
 *   out         device, bf16 [tovl_dispatch_rows(T,k,E)][N]: rows [off[e],
 *               off[e+1]) = dispatched rows x W[e]; padding rows are zero;
 *               rows >= off[E] are not written
 * Padding rows of `dispatched` are re-zeroed whenever the segment layout or
 * the buffer differs from the previous dispatch call on this handle.  An
 * expert id outside [0, E) makes the round a no-op that sets
 * TOVL_ERR_INVALID in the status word. */
int tovl_dispatch_grouped_gemm(tovl_handle h, const void* x, int T, int H, const int* topk_idx, int k, int E,
                               const void* W, int N, void* dispatched, int* expert_offsets, void* out,
                               void* stream);

/* GEMM + reduce-scatter over logical shards (a row-parallel layer: ReduceScatter
 * is the collective the platform page benchmarks beside AllGather, section
 * 3).  Shard s holds the K-slice X_s [M][Ks] of the activations and W_s
 * [Ks][N] of the weights; its partial P_s = X_s x W_s is computed by the
 * consumer CTAs (fp32 accumulation, rounded to bf16) and every partial tile
 * is published with the single-writer protocol: its epilogue warps arrive on
 * the tile's counter (acq_rel) once their stores are in global memory, and
 * the last arrival release-stores the sequence into the tile's slot.  The
 * reducers poll the S slots of an output tile (acquire) and write
 *   out[m][n] = bf16( sum_s f32(P_s[m][n]) ), fp32 sums in ascending s.
 * By default producer CTAs reduce; with option 19 = 1 (and no producer count
 * set) the reducer of output tile o is the CTA pair that computes shard
 * (o mod S)'s partial of it.
 *   X           device, bf16 [S][M][Ks]
 *   num_shards  S, 1..64
 *   M           rows, a multiple of 128
 *   Ks          multiple of 64, at most 32768
 *   W           device, bf16 [S][Ks][N], N a multiple of 256
 *   partials    device, bf16 [S][M][N]: receives P_s
 *   out         device, bf16 [M][N]: receives the reduced rows
 * Partial tiles (S x (M/128) x (N/256), or half that with CTA pairs) must
 * not exceed max_rows/64 x k_slices, the handle's counter capacity.  One
 * round (one sequence number). */
int tovl_gemm_reduce_scatter(tovl_handle h, const void* X, int num_shards, int M, int Ks, const void* W, int N,
                             void* partials, void* out, void* stream);

/* Combine: the reverse of the last dispatch round on this handle ("cross-GPU
 * sync protocols on PCIe", section 3, the layer-1 combine: every expert
 * output row goes back to its token's staging row; each 64-row staging chunk
 * is counted with acq_rel atomics and published by the elected last writer;
 * reducers poll the chunk slots with acquire loads).
 *   y           device, bf16 [rows][N]: expert outputs in the dispatched layout
 *               of the last tovl_dispatch_grouped_gemm call (its `out`)
 *   N           row length of y, multiple of 64, at most 32768
 *   gate_w      device, fp32 [T][k]: weight of pair (t, j)
 *   staging     device, bf16 [T*k][N]: receives staging[t*k + j] = y[dst(t, j)]
 *   combined    device, bf16 [T][N]: receives round-to-nearest-even of
 *               sum_j gate_w[t][j] * staging[t*k + j], every product and every
 *               partial sum rounded to fp32, j ascending
 *   stream      cudaStream_t, ordered after the dispatch call
 * T, k and the routing plan are the last dispatch call's; T*k <= max_rows.
 * Without an earlier dispatch on the handle the call returns
 * TOVL_ERR_INVALID; after a dispatch whose plan was rejected (bad expert id)
 * the round is a no-op that sets TOVL_ERR_INVALID in the status word; after
 * a dispatch round without tokens (T = 0) the call returns TOVL_OK and does
 * nothing (no round).  Otherwise one round (one sequence number), like the
 * other calls.  With option 18 on (the default) and no producer count set,
 * every CTA copies in 10 of its 16 warps and reduces in the other 6;
 * otherwise producer CTAs copy (option 1, default 7/12 of the SMs) and the
 * remaining SMs reduce. */
int tovl_combine(tovl_handle h, const void* y, int N, const float* gate_w, void* staging, void* combined,
                 void* stream);

/* ---------------------------------------------------------------- no-allocation plan
 * The pages have no counterpart to this entry point; it serves callers that
 * must not allocate device memory themselves (code inside another
 * framework's memory budget, latency-critical loops that cannot afford
 * cudaMalloc's device-wide synchronisation, plugins whose host owns every
 * allocation).
 *
 * tovl_dispatch_plan_noalloc computes the routing plan of a dispatch round
 * -- the same kernels and results as tovl_dispatch_grouped_gemm's plan --
 * without a handle and without allocating: its scratch is one fixed device
 * array inside the library (about 0.3 MB, held by every GPU that loads the
 * library until the process exits).
 *   topk_idx        device, int32 [T][k], expert of each pair in [0, E)
 *   expert_offsets  device, int32 [E+1]: padded segment starts (multiples of
 *                   128); all zero if an expert id is out of range (the only
 *                   report of that error: this entry point has no status word)
 *   dst_rows        device, int32 [T*k]: destination row of each pair, rows
 *                   of one expert in ascending (t, j) order; not written when
 *                   an expert id is out of range
 *   stream          cudaStream_t; the call is asynchronous
 * Limits: T*k <= TOVL_NOALLOC_MAX_PAIRS and E <= TOVL_NOALLOC_MAX_EXPERTS;
 * larger sizes return TOVL_ERR_UNSUPPORTED before anything is enqueued.
 * It runs on the calling thread's current device.  The first call on a
 * device looks up the scratch array's device address (cudaGetSymbolAddress)
 * and keeps it for the life of the process; make that first call before any
 * stream capture.  The kept address does not survive a reset of the device
 * (cudaDeviceReset, or a reset of its primary context): after one, this
 * entry point must not be called again in that process.  All calls
 * on a device share the one array and it keeps the previous call's
 * contents, so calls whose kernels overlap on the GPU (other streams, other
 * threads) race and must be serialised by the caller. */
#define TOVL_NOALLOC_MAX_PAIRS 32768
#define TOVL_NOALLOC_MAX_EXPERTS 64
int tovl_dispatch_plan_noalloc(const int* topk_idx, int T, int k, int E, int* expert_offsets, int* dst_rows,
                               void* stream);

/* ---------------------------------------------------------------- controls
 * The acceptance method of the platform page, section 5, compares the fused
 * kernel with its parts run alone on the same SM counts. */

/* GEMM-only control: the consumer CTAs of tovl_gather_gemm (same count C)
 * with gates disabled, on an already filled A.  A: device bf16 [M][K],
 * W: device bf16 [K][N], out: device bf16 [M][N].  Not a protocol round. */
int tovl_gemm_only(tovl_handle h, const void* A, int M, int K, const void* W, int N, void* out, void* stream);

/* Copy-only control: the producer CTAs of tovl_gather_gemm (same count P)
 * with the full protocol and no consumers.  Arguments as tovl_gather_gemm.
 * A protocol round. */
int tovl_copy_only(tovl_handle h, const void* const* shards, int num_shards, int rows_per_shard, int K,
                   void* gathered, void* stream);

/* Permuted row copy dst[perm[i]] = src[i] over 64-row destination chunks.
 *   src, dst    device, n_rows x row_bytes each (row_bytes multiple of 16)
 *   perm        device, int32 [n_rows], a permutation of [0, n_rows)
 *   gated       1: every row is an arrival on its destination chunk, the last
 *               arrival publishes the chunk slot, waiter CTAs observe the
 *               slots (a protocol round); 0: the same copy with no
 *               protocol (not a round)
 *   stamps      1: record publish and first-observe times per chunk
 *               (read them with tovl_read_latency)
 * The copy mechanism is the handle's copy mode (option 3): vector copies, bulk
 * copies (rows up to 24 KB; larger rows return TOVL_ERR_UNSUPPORTED), or the
 * default automatic choice by row size.  Results are identical in every mode. */
int tovl_gated_copy(tovl_handle h, const void* src, void* dst, long long n_rows, int row_bytes, const int* perm,
                    int gated, int stamps, void* stream);

/* ---------------------------------------------------------------- diagnostics */

/* Synchronises the handle's last stream, returns the sticky device status
 * (TOVL_OK if none) and clears it. */
int tovl_sync_status(tovl_handle h);

/* Lengths of the control-plane arrays: chunk slots/counters
 * (max_rows/64 chunks x k_slices, index chunk*k_slices + slice) and
 * row-block counters (max_rows/128 blocks x k_slices). */
int tovl_ctrl_sizes(tovl_handle h, int* n_chunks, int* n_blocks);

/* Copies the control plane to host arrays (after synchronising): slots and
 * cnts [n_chunks], rbcnts [n_blocks] (lengths from tovl_ctrl_sizes);
 * *seq = calls that were protocol rounds.
 * Any pointer may be NULL. */
int tovl_read_ctrl(tovl_handle h, int* slots, int* cnts, int* rbcnts, long long* seq);

/* Copies the last dispatch round's plan to host arrays (after
 * synchronising): counts [E], dst [T*k], src_of_dst [m_pad] (token of each
 * row, -1 for padding), pad [m_pad/128], blk_expert [m_pad/128], *m_pad.
 * Any pointer may be NULL. */
int tovl_read_plan(tovl_handle h, int* counts, int* dst, int* src_of_dst, int* pad, int* blk_expert, int* m_pad);

/* Options for sweeps: 1 = producer CTAs (0 = automatic split; reads back
 * the count the last call used), 2 = consumer CTAs, 3 = copy mode,
 * 4 = statistics on/off, 5 = wait timeout in ns, 6 = copy-sweep CTAs,
 * 7 = copy-sweep waiter CTAs, 9 = k_slices (read only),
 * 10 = CTA-pair consumers for gather calls (1 = on, the default: two CTAs of a
 * cluster compute a 256x256 tile with cta_group::2 MMAs; 0 = one CTA per
 * 128x256 tile; reads back 0 if the device cannot co-schedule pairs),
 * 11 = co-resident CTA pairs on the device (read only), 12 = 1 if
 * cooperative launches are accepted with pairs (read only), 13 = fused
 * launches request the cooperative co-residency guarantee (1, the default;
 * 0 launches the same kernel without it, for tools that cannot replay
 * cooperative launches -- the grid still fits one CTA per SM; the same
 * switch applies to the combine kernel and to gated copies),
 * 14 = producer copy path of the fused kernels: 0 = 16-byte vector loads and
 * stores through registers (the default), 1 = bulk asynchronous loads of each
 * row segment into a per-warp shared-memory buffer, then 16-byte vector
 * stores (results are identical),
 * 15 = programmatic dependent launch between the library's own kernels
 * (1, the default: a kernel's launch and prologue overlap the end of the
 * kernel before it -- plan counting, plan finalisation, the fused kernel,
 * combine -- and every kernel waits for its predecessor before it reads
 * memory; 0 = plain stream order; reads back 0 if the device refused it),
 * 16 = role switch (1, the default; 0 = fixed roles; 2 = also for CTA-pair
 * tiles): in tovl_dispatch_grouped_gemm with producer CTAs (option 18 = 0)
 * consumer tiles are handed out by a ticket counter and producer CTAs take
 * tiles once their copies are done
 * (the automatic split then gives the copy twice its balance share); with
 * 256-row segments this applies at 2 only (a CTA pair takes one ticket for
 * both CTAs; measured about 1 % slower than fixed pair roles on the uniform
 * and Zipf workloads, whose last wave the joining producers cannot fill); in
 * tovl_gemm_reduce_scatter consumer CTAs that have finished their partial
 * tiles take reduction items beside the producer CTAs,
 * 17 = expert segment alignment of tovl_dispatch_grouped_gemm in rows: 128
 * (the default: segments padded to the 128-row block, the layout the oracle
 * defines) or 256 (segments padded to two blocks, so CTA pairs compute
 * 256-row tiles inside one expert; the padded rows are zero and their
 * block counters are seeded like any padding; buffers then need
 * tovl_dispatch_rows_aligned(T, k, E, 256) rows; with embedded producers
 * CTA pairs run 128-row segments as well, two blocks of a segment per pair
 * tile, a segment's odd last block beside a phantom half that is computed
 * but never stored, so 256 no longer buys speed there),
 * 18 = embedded producers (1, the default: in tovl_dispatch_grouped_gemm and
 * tovl_combine;
 * 2 = also in tovl_gather_gemm; 0 = off): the call launches no producer
 * CTAs; every SM (every co-resident CTA pair) is a consumer and the
 * consumer CTAs' four spare warps copy the rows, in the producers' order and
 * with their counters and seeds (16-byte vector copies whatever option 14
 * says; the role switch does not apply; CTA pairs on 128-row segments, see
 * 17).  Measured on GB300: dispatch calls 16-17 % shorter than with
 * producer CTAs and single-CTA tiles (uniform 141.5 -> 118 us, Zipf 793 ->
 * 670 us), the TP gather 4-6 % slower (its three tile waves
 * stay three; the copy warps share the SMs),
 * 19 = where tovl_gemm_reduce_scatter sums the partials: 0 (the default) =
 * producer CTAs reduce, consumers join them when option 16 is on; 1 (when no
 * producer count is set) = every SM computes partial tiles and the CTA pair
 * that computes shard (o mod S)'s partial of output tile o sums that tile's S
 * partials in five otherwise idle warps, once all S partial tiles' slots are
 * published,
 * 20 = L2 eviction priorities of the fused calls' memory streams, a bit mask:
 * 1 producer source loads evict-last, 32 evict-first; 16 producer
 * destination stores evict-last; 4 A tensor loads evict-first; 8 weight
 * tensor loads evict-last; 2 output tensor stores evict-first; 0 = no
 * priorities; -1 (the default) = each call's measured choice: 32 | 8 for
 * tovl_gather_gemm, 8 for tovl_dispatch_grouped_gemm, 0 otherwise (results
 * are identical whatever the mask),
 * 23 = tile width of tovl_dispatch_grouped_gemm's CTA-pair tiles with
 * embedded producers (128- or 256-row segments): 1 (the default)
 * = 256 x 512 tiles when N is a multiple of 512 (one 512-column accumulator,
 * half the activation loads per MMA), else 256 x 256; 0 = always 256 x 256
 * (results agree within the GEMM tolerance either way),
 * 8 = fault injection for tests: consumer gates
 * wait for sequence seq + value, which no producer publishes, so every gate
 * expires after the wait timeout and the call ends with TOVL_ERR_TIMEOUT in
 * the status word (0 = off). */
int tovl_set_option(tovl_handle h, int option, long long value);
int tovl_get_option(tovl_handle h, int option, long long* value);

/* Statistics of the last call with statistics on: [0] gate polls,
 * [1] earliest consumer start ns, [2] latest consumer end ns, [3] earliest
 * producer start ns, [4] latest producer end ns. */
int tovl_read_stats(tovl_handle h, unsigned long long* stats, int n);

/* Timeline of the last fused call made with statistics on (%globaltimer ns):
 *   what 0: publish time of each chunk slice [n_chunks], index chunk*k_slices + slice
 *           (0 where no producer thread published it)
 *   what 1: time the consumer's gate passed each (tile, slice) [tiles*k_slices]
 *   what 2: time each tile's output was stored [tiles]
 *   what 3: time each tile's accumulator was complete (epilogue start) [tiles]
 * Tiles are numbered row block * (N/256) + column block; for dispatch calls
 * the tile count is the bound tovl_dispatch_rows/128 * N/256 (unused tiles
 * read 0), with 512-column pair tiles (option 23) N/512 column blocks.
 * n must not exceed the stated length. */
int tovl_read_trace(tovl_handle h, int what, long long* out, long long n);

/* Publish and first-observe %globaltimer stamps of the first n chunks of the
 * last stamped tovl_gated_copy. */
int tovl_read_latency(tovl_handle h, long long* pub_ns, long long* obs_ns, int n);

/* Number of SMs of the handle's device. */
int tovl_num_sms(tovl_handle h);

const char* tovl_error_string(int code);

/* Text of the last CUDA error seen by this handle ("" if none). */
const char* tovl_last_error(tovl_handle h);

#ifdef __cplusplus
}
#endif

#endif /* TOVL_H */
