// tovl_api.cu -- host implementation of the C ABI declared in include/tovl.h.
//
// Owns the control plane of a handle (slots, counters, status word, plan
// scratch) and the per-handle sequence number; validates every argument on
// the host; encodes TMA tensor maps; launches the kernels on the caller's
// stream.  No device work runs here besides memsets at creation.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <new>

#include "tovl.h"
#include "ctrl.cuh"
#include "launch.cuh"

#define TOVL_API extern "C" __attribute__((visibility("default")))

using namespace tovl;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct tovl_ctx {
    tovl_config cfg;
    int device = 0;
    int num_sms = 0;
    int producers = 0;       // 0 = automatic split per call
    int last_P = 0, last_C = 0;
    int consumers = 0;
    int copy_mode = TOVL_COPY_AUTO;     // vector below 8 KB rows, bulk from 8 KB (measured best per size)
    int stats = 0;
    long long timeout_ns = 2000000000LL;
    int copy_ctas = 0;       // copy sweep copiers (0 = auto)
    int copy_waiters = 0;    // copy sweep waiters (0 = auto)
    int fault_gate_offset = 0;  // test hook: gates wait for seq + offset
    int slices = 1;          // K-slices per chunk watermark (fixed per handle)
    int pair_mode = 1;       // gather calls use CTA-pair (cta_group::2) consumers when possible
    int max_pairs = 0;       // co-resident CTA pairs of the pair kernel on this device
    bool coop_pairs = true;  // cooperative launch accepted together with clusters
    bool coop_enabled = true;  // fused launches ask for the co-residency guarantee
    int producer_mode = 0;     // fused producers: 0 vector copies, 1 staged bulk loads
    int dispatch_align = kBlockRows;  // expert segment alignment: 128, or 256 for CTA-pair tiles
    bool pdl = true;           // programmatic dependent launch between this library's kernels
    int role_switch = 1;       // 1: dispatch (single-CTA tiles) and reduce-scatter roles switch; 2: CTA-pair dispatch too
    int embedded = 1;          // without producer CTAs, the consumer CTAs' spare warps copy: 1 dispatch, 2 also gather
    int rs_epi = 0;            // 1: reduce-scatter tiles are summed by their owners' idle warps (no producer CTAs)
    int wide_tiles = 1;        // 1: CTA-pair dispatch tiles (embedded producers) are 256 x 512 where N allows
    int l2_hints = -1;         // kHint* bits for every fused call; -1 = each call's measured default
    bool pdl_ok = true;        // cleared if the device rejects the launch attribute
    long long seq = 0;
    Ctrl ctrl{};
    Plan plan{};
    int max_seg = 0;
    void* ctrl_mem = nullptr;    // one allocation for the control plane
    void* plan_mem = nullptr;    // one allocation for plan scratch
    cudaStream_t last_stream = nullptr;
    const void* last_dispatched = nullptr;
    int last_T = 0, last_k = 0, last_E = 0;
    long long last_tiles = 0;    // tiles and K-slices of the last fused call (trace layout)
    int last_ks = 0;
    EncodeTiledFn encode = nullptr;
    char last_error[256] = {0};
};

static int cuda_fail(tovl_ctx* h, cudaError_t e, const char* what)
{
    if (h) std::snprintf(h->last_error, sizeof h->last_error, "%s: %s", what, cudaGetErrorString(e));
    return TOVL_ERR_CUDA;
}

static bool aligned16(const void* p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

static long long ceil_div(long long a, long long b)
{
    return (a + b - 1) / b;
}

TOVL_API void tovl_default_config(tovl_config* cfg, int device)
{
    if (!cfg) return;
    std::memset(cfg, 0, sizeof *cfg);
    cfg->device = device;
    cfg->chunk_rows = kChunkRows;
    cfg->gate_rows = kBlockRows;
    cfg->producer_ctas = 0;
    cfg->consumer_ctas = 0;
    cfg->wait_timeout_ns = 0;
    cfg->copy_mode = TOVL_COPY_AUTO;
    cfg->max_rows = 1 << 16;
    cfg->max_pairs = 1 << 16;
    cfg->max_experts = 64;
    cfg->k_slices = 1;
}

TOVL_API const char* tovl_error_string(int code)
{
    switch (code) {
    case TOVL_OK: return "ok";
    case TOVL_ERR_INVALID: return "invalid argument";
    case TOVL_ERR_UNSUPPORTED: return "unsupported shape or device";
    case TOVL_ERR_CUDA: return "CUDA runtime error";
    case TOVL_ERR_TIMEOUT: return "device wait timed out";
    case TOVL_ERR_OOM: return "out of device memory";
    default: return "unknown error";
    }
}

TOVL_API const char* tovl_last_error(tovl_handle h)
{
    return h ? h->last_error : "";
}

TOVL_API long long tovl_dispatch_rows_aligned(int T, int k, int E, int align)
{
    if (T < 0 || k < 0 || E < 0 || (align != kBlockRows && align != 2 * kBlockRows)) return 0;
    return ceil_div(static_cast<long long>(T) * k + static_cast<long long>(E) * (align - 1), align) * align;
}

TOVL_API long long tovl_dispatch_rows(int T, int k, int E)
{
    return tovl_dispatch_rows_aligned(T, k, E, kBlockRows);
}

static void free_all(tovl_ctx* h)
{
    if (h->ctrl_mem) cudaFree(h->ctrl_mem);
    if (h->plan_mem) cudaFree(h->plan_mem);
    h->ctrl_mem = h->plan_mem = nullptr;
}

// Bump allocator over one device allocation; every piece 256-byte aligned.
struct Carve {
    char* base;
    size_t off;
    template <class T>
    T* take(size_t n)
    {
        off = (off + 255) & ~static_cast<size_t>(255);
        T* p = reinterpret_cast<T*>(base ? base + off : nullptr);
        off += n * sizeof(T);
        return p;
    }
};

static void carve_ctrl(Carve& c, Ctrl& ctrl, int n_chunks, int n_blocks, int S)
{
    ctrl.slot = c.take<int>(static_cast<size_t>(n_chunks) * S);
    ctrl.cnt = c.take<int>(static_cast<size_t>(n_chunks) * S);
    ctrl.rbcnt = c.take<int>(static_cast<size_t>(n_blocks) * S);
    ctrl.status = c.take<int>(1);
    ctrl.abort_seq = c.take<int>(1);
    ctrl.work = c.take<int>(1);
    ctrl.stats = c.take<unsigned long long>(kNumStats);
    ctrl.pub_ns = c.take<long long>(static_cast<size_t>(n_chunks) * S);
    ctrl.obs_ns = c.take<long long>(n_chunks);
    ctrl.trace = c.take<long long>(kTraceCap);
    ctrl.trace_cap = kTraceCap;
    ctrl.n_chunk_cap = n_chunks;
    ctrl.n_block_cap = n_blocks;
    ctrl.n_slices = S;
}

static void carve_plan(Carve& c, Plan& p, int E, int max_seg, int max_pairs, long long rows, int n_blocks)
{
    p.counts = c.take<int>(E);
    p.off = c.take<int>(E + 1);
    p.prev_off = c.take<int>(E + 1);
    p.seg_count = c.take<int>(static_cast<size_t>(max_seg) * E);
    p.local_rank = c.take<int>(max_pairs);
    p.dst = c.take<int>(max_pairs);
    p.src_of_dst = c.take<int>(rows);
    p.pad = c.take<int>(n_blocks);
    p.blk_expert = c.take<int>(n_blocks);
    p.meta = c.take<int>(4);
    p.pair_tab = c.take<int>(static_cast<size_t>(n_blocks) + 1);
}

TOVL_API int tovl_create(tovl_handle* out, const tovl_config* cfg_in)
{
    if (!out) return TOVL_ERR_INVALID;
    *out = nullptr;
    if (!cfg_in) return TOVL_ERR_INVALID;
    tovl_config cfg = *cfg_in;
    if (cfg.chunk_rows == 0) cfg.chunk_rows = kChunkRows;
    if (cfg.gate_rows == 0) cfg.gate_rows = kBlockRows;
    if (cfg.chunk_rows != kChunkRows || cfg.gate_rows != kBlockRows) return TOVL_ERR_UNSUPPORTED;
    if (cfg.max_rows < 1 || cfg.max_rows > (1LL << 30)) return TOVL_ERR_INVALID;
    if (cfg.max_pairs < 0 || cfg.max_pairs > (1 << 28)) return TOVL_ERR_INVALID;
    if (cfg.max_experts < 0 || cfg.max_experts > kMaxExperts) return TOVL_ERR_INVALID;
    if (cfg.producer_ctas < 0 || cfg.consumer_ctas < 0 || cfg.wait_timeout_ns < 0) return TOVL_ERR_INVALID;
    if (cfg.copy_mode != TOVL_COPY_VECTOR && cfg.copy_mode != TOVL_COPY_BULK && cfg.copy_mode != TOVL_COPY_AUTO)
        return TOVL_ERR_INVALID;
    if (cfg.k_slices == 0) cfg.k_slices = 1;
    if (cfg.k_slices < 1 || cfg.k_slices > kMaxSlices) return TOVL_ERR_INVALID;

    int n_dev = 0;
    if (cudaGetDeviceCount(&n_dev) != cudaSuccess || n_dev == 0) {
        cudaGetLastError();
        return TOVL_ERR_UNSUPPORTED;
    }
    if (cfg.device < 0 || cfg.device >= n_dev) return TOVL_ERR_INVALID;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, cfg.device) != cudaSuccess) return TOVL_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return TOVL_ERR_UNSUPPORTED;

    tovl_ctx* h = new (std::nothrow) tovl_ctx();
    if (!h) return TOVL_ERR_OOM;
    h->cfg = cfg;
    h->device = cfg.device;
    h->num_sms = prop.multiProcessorCount;
    h->producers = cfg.producer_ctas;
    h->consumers = cfg.consumer_ctas;
    h->copy_mode = cfg.copy_mode;
    h->slices = cfg.k_slices;
    if (cfg.wait_timeout_ns) h->timeout_ns = cfg.wait_timeout_ns;

    int prev_dev = 0;
    cudaGetDevice(&prev_dev);
    cudaError_t e = cudaSetDevice(h->device);
    if (e != cudaSuccess) {
        delete h;
        return TOVL_ERR_CUDA;
    }
    int rc = TOVL_OK;
    do {
        if ((e = prepare_fused()) != cudaSuccess) { rc = cuda_fail(h, e, "prepare fused"); break; }
        if ((e = prepare_plan()) != cudaSuccess) { rc = cuda_fail(h, e, "prepare plan"); break; }
        if ((e = prepare_copy()) != cudaSuccess) { rc = cuda_fail(h, e, "prepare copy"); break; }
        if ((e = prepare_combine()) != cudaSuccess) { rc = cuda_fail(h, e, "prepare combine"); break; }
        if (fused_max_active_per_sm() < 1) { rc = TOVL_ERR_UNSUPPORTED; break; }
        h->max_pairs = fused_max_active_pairs();

        const int n_chunks = static_cast<int>(ceil_div(cfg.max_rows, kChunkRows));
        const int n_blocks = static_cast<int>(ceil_div(cfg.max_rows, kBlockRows));
        Carve sizing{nullptr, 0};
        Ctrl tmp_ctrl{};
        carve_ctrl(sizing, tmp_ctrl, n_chunks, n_blocks, h->slices);
        const size_t ctrl_bytes = sizing.off + 256;
        if ((e = cudaMalloc(&h->ctrl_mem, ctrl_bytes)) != cudaSuccess) { rc = TOVL_ERR_OOM; cudaGetLastError(); break; }
        if ((e = cudaMemset(h->ctrl_mem, 0, ctrl_bytes)) != cudaSuccess) { rc = cuda_fail(h, e, "memset"); break; }
        Carve cc{static_cast<char*>(h->ctrl_mem), 0};
        carve_ctrl(cc, h->ctrl, n_chunks, n_blocks, h->slices);

        const int E = cfg.max_experts > 0 ? cfg.max_experts : 1;
        h->max_seg = static_cast<int>(ceil_div(cfg.max_pairs > 0 ? cfg.max_pairs : 1, 1024));
        Carve psz{nullptr, 0};
        Plan tmp_plan{};
        carve_plan(psz, tmp_plan, E, h->max_seg, cfg.max_pairs > 0 ? cfg.max_pairs : 1, cfg.max_rows, n_blocks);
        const size_t plan_bytes = psz.off + 256;
        if ((e = cudaMalloc(&h->plan_mem, plan_bytes)) != cudaSuccess) { rc = TOVL_ERR_OOM; cudaGetLastError(); break; }
        if ((e = cudaMemset(h->plan_mem, 0, plan_bytes)) != cudaSuccess) { rc = cuda_fail(h, e, "memset"); break; }
        Carve pc{static_cast<char*>(h->plan_mem), 0};
        carve_plan(pc, h->plan, E, h->max_seg, cfg.max_pairs > 0 ? cfg.max_pairs : 1, cfg.max_rows, n_blocks);

        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
            rc = cuda_fail(h, e == cudaSuccess ? cudaErrorSymbolNotFound : e, "cuTensorMapEncodeTiled");
            break;
        }
        h->encode = reinterpret_cast<EncodeTiledFn>(fn);
        if ((e = cudaDeviceSynchronize()) != cudaSuccess) { rc = cuda_fail(h, e, "create sync"); break; }
    } while (0);
    if (rc != TOVL_OK) {
        free_all(h);
        delete h;
        cudaSetDevice(prev_dev);
        return rc;
    }
    cudaSetDevice(prev_dev);
    *out = h;
    return TOVL_OK;
}

TOVL_API int tovl_destroy(tovl_handle h)
{
    if (!h) return TOVL_OK;
    int prev_dev = 0;
    cudaGetDevice(&prev_dev);
    cudaSetDevice(h->device);
    if (h->last_stream) cudaStreamSynchronize(h->last_stream);
    cudaDeviceSynchronize();
    free_all(h);
    cudaSetDevice(prev_dev);
    delete h;
    return TOVL_OK;
}

TOVL_API int tovl_num_sms(tovl_handle h)
{
    return h ? h->num_sms : 0;
}

// 2-D bf16 tensor map: `inner` contiguous elements per row, `outer` rows,
// rows `stride` bytes apart; boxes of box_inner x box_outer, 128B swizzle,
// out-of-range elements read as zero.
static int encode_2d(tovl_ctx* h, CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                     uint64_t stride, uint32_t box_inner, uint32_t box_outer,
                     CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B)
{
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {stride};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = h->encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                                 estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        std::snprintf(h->last_error, sizeof h->last_error, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
        return TOVL_ERR_INVALID;
    }
    return TOVL_OK;
}

// Weights W [rows][N] bf16 (N contiguous, N a multiple of 64) as a 3-D map
// [N/64][rows][64]: one load brings kWBlocks 64-column blocks of 64 rows, in
// the shared-memory layout of kWBlocks separate 64 x 64 boxes.
static int encode_weights(tovl_ctx* h, CUtensorMap* map, const void* W, uint64_t N, uint64_t rows)
{
    cuuint64_t dims[3] = {64, rows, N / 64};
    cuuint64_t strides[2] = {N * 2, 128};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kTileK), static_cast<cuuint32_t>(kWBlocks)};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = h->encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(W), dims, strides, box,
                                 estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        std::snprintf(h->last_error, sizeof h->last_error, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
        return TOVL_ERR_INVALID;
    }
    return TOVL_OK;
}

// Weights for 256 x 512 CTA-pair tiles: the [rows][N] matrix viewed as
// [N/256][4][rows][64] (64-column blocks grouped by 256-column half), box
// 64 x 64 x 2 x 2: one load brings a CTA's 128 columns of both halves of a
// 512-column tile for one k-block.
static int encode_weights_wide(tovl_ctx* h, CUtensorMap* map, const void* W, uint64_t N, uint64_t rows)
{
    cuuint64_t dims[4] = {64, rows, kTileN / 64, N / kTileN};
    cuuint64_t strides[3] = {N * 2, 128, kTileN * 2};
    cuuint32_t box[4] = {64, static_cast<cuuint32_t>(kTileK), 2, 2};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = h->encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(W), dims, strides, box,
                                 estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        std::snprintf(h->last_error, sizeof h->last_error, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
        return TOVL_ERR_INVALID;
    }
    return TOVL_OK;
}

// Waits inside one CTA's own pipeline depend on its gate waits, so their
// bound must outlast a gate timeout.
static long long pipe_timeout(const tovl_ctx* h)
{
    return 4 * h->timeout_ns + 100000000LL;
}

static void base_params(tovl_ctx* h, FusedParams& p)
{
    std::memset(&p, 0, sizeof p);
    p.timeout_ns = h->timeout_ns;
    p.pipe_timeout_ns = pipe_timeout(h);
    p.stats = h->stats;
    p.producer_mode = h->producer_mode;
    p.l2_hints = h->l2_hints > 0 ? h->l2_hints : 0;
    p.ctrl = h->ctrl;
}

// A call's L2 eviction hints when the handle leaves them to the call
// (option 20 = -1).  Measured on GB300 in interleaved A/B runs: weights
// evict-last shortens the uniform dispatch by 2 us and the Zipf dispatch by
// 10 us of 670; for the TP gather, shard loads evict-first (read once) with
// weights evict-last takes 0.9 us off the fused call.
static void default_hints(const tovl_ctx* h, FusedParams& p, int hints)
{
    if (h->l2_hints < 0) p.l2_hints = hints;
}

// Producer / consumer CTA split for one call.  With no fixed producer count,
// P balances the copy against the GEMM using per-SM rates measured for these
// kernels on GB300 (about 60 GB/s of copy traffic per producer SM, about
// 10 TFLOP/s per consumer SM), then grows while the consumers still finish
// the tiles in the same number of waves (section 4 of the platform page: SMs
// given to communication are taken from the GEMM, so the split is swept).
// With CTA pairs (pair = 2) a consumer unit is two CTAs computing 256-row
// tiles, both counts are even, and the grid is limited to the pairs that can
// be co-resident.
// With `joining` producers (they turn consumer once their copies are done),
// the copy only has to stay ahead of the GEMM: any P above the balance point
// gives about the same total, and a margin opens the gates sooner, so P is
// twice the balance point (measured on the dispatch workloads: flat between
// 1.5x and 3x) and the wave rule does not apply.
static void split_ctas(tovl_ctx* h, int& P, int& C, int n_mb, int n_nb, double copy_bytes, double flops, int pair,
                       bool joining = false)
{
    int S = h->num_sms;
    if (pair == 2 && 2 * h->max_pairs < S) S = 2 * h->max_pairs;
    const long long tiles = static_cast<long long>((n_mb + pair - 1) / pair) * n_nb;   // per consumer unit
    if (h->producers > 0) {
        P = h->producers < S - pair ? h->producers : S - pair;
    } else {
        const double tc = copy_bytes / 60e9, tg = flops / 10e12;
        int p = static_cast<int>(S * tc / (tc + tg + 1e-30) + 0.5);
        const int pmax = joining ? S / 2 : S / 4;
        if (joining) p *= 2;
        p = p < 4 ? 4 : (p > pmax ? pmax : p);
        if (tiles > 0 && !joining) {
            const int units = (S - p) / pair;
            const long long waves = (tiles + units - 1) / units;
            const int cmin = static_cast<int>((tiles + waves - 1) / waves) * pair;
            if (S - cmin > p) p = S - cmin < pmax ? S - cmin : pmax;
        }
        P = p;
    }
    if (pair == 2) P = (P + 1) & ~1;
    C = h->consumers ? h->consumers : S - P;
    if (C > S - P) C = S - P;
    if (pair == 2) C &= ~1;
    if (C < pair) C = pair;
    h->last_P = P;
    h->last_C = C;
}

// Launch with the cooperative guarantee of co-residency; a device that does
// not accept it together with a cluster shape is launched without it (the
// grid still fits: one CTA per SM, at most the co-resident pairs).
static cudaError_t launch(tovl_ctx* h, const FusedParams& p, cudaStream_t s, bool cooperative, int pair)
{
    if (pair == 2 && !h->coop_pairs) cooperative = false;
    if (!h->coop_enabled) cooperative = false;
    bool pdl = h->pdl && h->pdl_ok;
    cudaError_t e = launch_fused(p, s, cooperative, pair, pdl);
    if (e != cudaSuccess && pdl) {
        cudaGetLastError();
        pdl = false;
        e = launch_fused(p, s, cooperative, pair, false);
        if (e == cudaSuccess) h->pdl_ok = false;
    }
    if (e != cudaSuccess && pair == 2 && cooperative) {
        cudaGetLastError();
        e = launch_fused(p, s, false, pair, pdl);
        if (e == cudaSuccess) h->coop_pairs = false;
    }
    return e;
}

// Slicing and producer-item geometry of one call: k_slices never exceeds the
// K-blocks; an item moves item_rows rows of one slice, at most 8 KB per pass;
// the producers' ordering group is the consumers' first wave of row blocks.
static void call_geometry(const tovl_ctx* h, FusedParams& p, int C, int pair)
{
    p.k_slices = h->slices < p.n_kb ? h->slices : p.n_kb;
    const int max_kbs = (p.n_kb + p.k_slices - 1) / p.k_slices;
    const int n16 = max_kbs * kTileK * 2 / 16;
    int ri = 64;
    while (ri > 1 && ri * n16 > kItemInt4) ri >>= 1;
    p.item_rows = ri;
    const int units = C / pair;
    p.wave_blocks = units > 0 ? (units + p.n_nb - 1) / p.n_nb * pair : 1;
    if (p.wave_blocks < 1) p.wave_blocks = 1;
}

static int reset_stats(tovl_ctx* h, cudaStream_t s, long long tiles, int ks)
{
    h->last_tiles = tiles;
    h->last_ks = ks;
    if (!h->stats) return TOVL_OK;
    // min slots start at all-ones, the others at zero; the timeline at zero
    cudaError_t e = cudaMemsetAsync(h->ctrl.stats, 0, kNumStats * sizeof(unsigned long long), s);
    long long n_trace = tiles * (ks + 2);
    if (n_trace > h->ctrl.trace_cap) n_trace = h->ctrl.trace_cap;
    if (e == cudaSuccess && n_trace > 0) e = cudaMemsetAsync(h->ctrl.trace, 0, n_trace * sizeof(long long), s);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(h->ctrl.pub_ns, 0,
                            static_cast<size_t>(h->ctrl.n_chunk_cap) * h->ctrl.n_slices * sizeof(long long), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->ctrl.stats + kStatConsStartNs, 0xff, sizeof(unsigned long long), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->ctrl.stats + kStatProdStartNs, 0xff, sizeof(unsigned long long), s);
    return e == cudaSuccess ? TOVL_OK : cuda_fail(h, e, "stats reset");
}

struct DeviceGuard {
    int prev = 0;
    explicit DeviceGuard(int dev)
    {
        cudaGetDevice(&prev);
        if (prev != dev) cudaSetDevice(dev);
    }
    ~DeviceGuard() { cudaSetDevice(prev); }
};

// Shared validation of the gather shapes.
static int check_gather(tovl_ctx* h, const void* const* shards, int S, int R, int K)
{
    if (!shards || S < 1 || S > kMaxShards || R < 1 || K < kTileK || K % kTileK) return TOVL_ERR_INVALID;
    if (K > kMaxK) return TOVL_ERR_UNSUPPORTED;
    if (static_cast<long long>(S) * R > h->cfg.max_rows) return TOVL_ERR_INVALID;
    for (int s = 0; s < S; ++s)
        if (!shards[s] || !aligned16(shards[s])) return TOVL_ERR_INVALID;
    return TOVL_OK;
}

// flags: 1 = producers, 2 = consumers, 4 = gated
static int run_gather(tovl_handle h, const void* const* shards, int S, int R, int K, const void* W, int N,
                      void* gathered, const void* A, void* out, cudaStream_t stream, int flags)
{
    const int M = S * R;
    FusedParams p;
    base_params(h, p);
    p.mode = kModeGather;
    p.M = M;
    p.N = N;
    p.K = K;
    p.n_kb = K / kTileK;
    p.n_nb = N / kTileN;
    p.row_bytes = K * 2;
    // the split (and with it P for copy-only and C for GEMM-only) and the
    // kernel shape are the ones the fused call uses, so the controls run
    // under the same launch (shared-memory size, and with it the producer
    // SMs' L1 share)
    const int pair = (h->pair_mode && h->max_pairs > 0) ? 2 : 1;
    const int split_pair = pair;
    const int n_mb = (M + kTileM - 1) / kTileM;
    int P, C;
    split_ctas(h, P, C, n_mb, p.n_nb, 4.0 * M * K, 2.0 * M * static_cast<double>(N) * K, split_pair);
    p.n_producers = (flags & 1) ? P : 0;
    p.n_consumers = (flags & 2) ? C : 0;
    p.gated = (flags & 4) ? 1 : 0;
    if (h->embedded == 2 && flags == (1 | 2 | 4)) {
        // the fused call without producer CTAs: every SM (co-resident pair)
        // a consumer, the copy in the consumer CTAs' spare warps
        C = (pair == 2 && 2 * h->max_pairs < h->num_sms) ? 2 * h->max_pairs : h->num_sms;
        if (h->consumers > 0 && h->consumers < C) C = h->consumers;
        if (pair == 2) C &= ~1;
        P = 0;
        h->last_P = P;
        h->last_C = C;
        p.n_producers = 0;
        p.n_consumers = C;
        p.embedded = 1;
    }
    call_geometry(h, p, C, split_pair);
    default_hints(h, p, kHintSrcFirst | kHintBLast);
    p.n_shards = S;
    p.rows_per_shard = R;
    for (int s = 0; s < S; ++s) p.shard[s] = shards ? shards[s] : nullptr;
    p.gathered = gathered;
    p.out = out;
    p.out_rows = M;
    int rc;
    if (flags & 2) {
        if ((rc = encode_2d(h, &p.tmap_a, A, K, M, static_cast<uint64_t>(K) * 2, kTileK, kTileM)) != TOVL_OK) return rc;
        if ((rc = encode_weights(h, &p.tmap_b, W, N, K)) != TOVL_OK) return rc;
        if ((rc = encode_2d(h, &p.tmap_out, out, N, M, static_cast<uint64_t>(N) * 2, kEpiBoxCols, 32,
                            CU_TENSOR_MAP_SWIZZLE_64B)) != TOVL_OK)
            return rc;
    }
    const bool round = (flags & 1) != 0;
    if (round) p.seq = static_cast<int>(h->seq + 1);
    else p.seq = static_cast<int>(h->seq);
    p.gate_seq = p.seq + h->fault_gate_offset;
    p.trace_tiles = (flags & 2) ? (n_mb + pair - 1) / pair * p.n_nb : 0;
    if ((rc = reset_stats(h, stream, p.trace_tiles, p.k_slices)) != TOVL_OK) return rc;
    const cudaError_t e = launch(h, p, stream, (flags & 4) != 0, pair);
    if (e != cudaSuccess) return cuda_fail(h, e, "fused launch");
    if (round) h->seq += 1;
    h->last_stream = stream;
    return TOVL_OK;
}

TOVL_API int tovl_gather_gemm(tovl_handle h, const void* const* shards, int num_shards, int rows_per_shard, int K,
                              const void* W, int N, void* gathered, void* out, void* stream)
{
    if (!h) return TOVL_ERR_INVALID;
    int rc = check_gather(h, shards, num_shards, rows_per_shard, K);
    if (rc != TOVL_OK) return rc;
    if (!W || !gathered || !out || !aligned16(W) || !aligned16(gathered) || !aligned16(out)) return TOVL_ERR_INVALID;
    if (N < kTileN || N % kTileN) return TOVL_ERR_UNSUPPORTED;
    DeviceGuard g(h->device);
    return run_gather(h, shards, num_shards, rows_per_shard, K, W, N, gathered, gathered, out,
                      static_cast<cudaStream_t>(stream), 1 | 2 | 4);
}

TOVL_API int tovl_copy_only(tovl_handle h, const void* const* shards, int num_shards, int rows_per_shard, int K,
                            void* gathered, void* stream)
{
    if (!h) return TOVL_ERR_INVALID;
    int rc = check_gather(h, shards, num_shards, rows_per_shard, K);
    if (rc != TOVL_OK) return rc;
    if (!gathered || !aligned16(gathered)) return TOVL_ERR_INVALID;
    DeviceGuard g(h->device);
    return run_gather(h, shards, num_shards, rows_per_shard, K, nullptr, kTileN, gathered, nullptr, nullptr,
                      static_cast<cudaStream_t>(stream), 1);
}

TOVL_API int tovl_gemm_only(tovl_handle h, const void* A, int M, int K, const void* W, int N, void* out, void* stream)
{
    if (!h) return TOVL_ERR_INVALID;
    if (!A || !W || !out || !aligned16(A) || !aligned16(W) || !aligned16(out)) return TOVL_ERR_INVALID;
    if (M < 1 || K < kTileK || K % kTileK) return TOVL_ERR_INVALID;
    if (N < kTileN || N % kTileN) return TOVL_ERR_UNSUPPORTED;
    DeviceGuard g(h->device);
    return run_gather(h, nullptr, 1, M, K, W, N, nullptr, A, out, static_cast<cudaStream_t>(stream), 2);
}

TOVL_API int tovl_dispatch_grouped_gemm(tovl_handle h, const void* x, int T, int H, const int* topk_idx, int k, int E,
                                        const void* W, int N, void* dispatched, int* expert_offsets, void* out,
                                        void* stream)
{
    if (!h) return TOVL_ERR_INVALID;
    // a round without tokens (T = 0) reads neither x nor topk_idx
    if (((!x || !topk_idx) && T > 0) || !W || !dispatched || !expert_offsets || !out) return TOVL_ERR_INVALID;
    if (!aligned16(x) || !aligned16(W) || !aligned16(dispatched) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(topk_idx) & 3u) || (reinterpret_cast<uintptr_t>(expert_offsets) & 3u))
        return TOVL_ERR_INVALID;
    if (T < 0 || k < 1 || E < 1 || E > h->cfg.max_experts || E > kMaxExperts) return TOVL_ERR_INVALID;
    if (H < kTileK || H % kTileK) return TOVL_ERR_INVALID;
    if (H > kMaxK) return TOVL_ERR_UNSUPPORTED;
    if (N < kTileN || N % kTileN) return TOVL_ERR_UNSUPPORTED;
    const long long pairs = static_cast<long long>(T) * k;
    if (pairs > h->cfg.max_pairs) return TOVL_ERR_INVALID;
    const int align = h->dispatch_align;
    const long long rows = tovl_dispatch_rows_aligned(T, k, E, align);
    if (rows > h->cfg.max_rows) return TOVL_ERR_INVALID;
    // 256-row segments let a CTA pair take two row blocks of one expert; with
    // 128-row segments and embedded producers CTA pairs take the plan's pair
    // tiles (two blocks of one segment, or one and a phantom half)
    const bool pair_ok = h->pair_mode && h->max_pairs > 0;
    const bool pair_tab = pair_ok && align == kBlockRows && h->embedded != 0;
    const int pair = (pair_ok && (align == 2 * kBlockRows || pair_tab)) ? 2 : 1;
    // CTA-pair tiles of the embedded-producer kernel 512 columns wide: half
    // the activation loads per MMA and one weight load per k-block for twice
    // the MMAs
    const bool wide = pair == 2 && h->embedded != 0 && h->wide_tiles != 0 && N % (2 * kTileN) == 0;
    DeviceGuard g(h->device);
    const cudaStream_t s = static_cast<cudaStream_t>(stream);

    PlanParams pp;
    std::memset(&pp, 0, sizeof pp);
    pp.topk = topk_idx;
    pp.n_pairs = static_cast<int>(pairs);
    pp.k = k;
    pp.E = E;
    pp.n_seg = static_cast<int>(ceil_div(pairs, 1024));
    pp.row_cap = static_cast<int>(rows);
    pp.block_cap = h->ctrl.n_block_cap;
    pp.force_zero = (dispatched != h->last_dispatched) ? 1 : 0;
    pp.expert_offsets = expert_offsets;
    pp.plan = h->plan;
    pp.status = h->ctrl.status;
    pp.work = h->ctrl.work;
    pp.align = align;
    cudaError_t e = launch_plan(pp, s, h->pdl && h->pdl_ok);
    if (e != cudaSuccess && h->pdl && h->pdl_ok) {
        cudaGetLastError();
        h->pdl_ok = false;
        e = launch_plan(pp, s, false);
    }
    if (e != cudaSuccess) return cuda_fail(h, e, "plan launch");

    FusedParams p;
    base_params(h, p);
    p.mode = kModeDispatch;
    p.M = static_cast<int>(rows);
    p.N = N;
    p.K = H;
    p.n_kb = H / kTileK;
    p.n_nb = N / (wide ? 2 * kTileN : kTileN);
    p.wide = wide ? 1 : 0;
    p.row_bytes = H * 2;
    int P, C;
    // role switch: consumer tiles (single-CTA or CTA-pair) come from the
    // ticket counter (zeroed by the plan kernel) and producer CTAs (pairs)
    // take tiles once their copies are done
    const bool emb = h->embedded != 0;
    const bool dyn = !emb && (pair == 1 ? h->role_switch != 0 : h->role_switch == 2);
    if (emb) {
        // every SM a consumer (CTA pairs: every co-resident pair); the copy
        // runs in the consumer CTAs' spare warps
        P = 0;
        C = (pair == 2 && 2 * h->max_pairs < h->num_sms) ? 2 * h->max_pairs : h->num_sms;
        if (h->consumers > 0 && h->consumers < C) C = h->consumers;
        if (pair == 2) C &= ~1;
        h->last_P = P;
        h->last_C = C;
    } else {
        split_ctas(h, P, C, static_cast<int>(rows / kTileM), p.n_nb, 4.0 * pairs * H,
                   2.0 * pairs * static_cast<double>(N) * H, pair, dyn);
    }
    p.n_producers = P;
    p.n_consumers = C;
    p.gated = 1;
    p.dyn = dyn ? 1 : 0;
    p.join = dyn ? 1 : 0;
    p.embedded = emb ? 1 : 0;
    call_geometry(h, p, C, pair);
    default_hints(h, p, kHintBLast);
    p.x = x;
    p.src_of_dst = h->plan.src_of_dst;
    p.pad = h->plan.pad;
    p.blk_expert = h->plan.blk_expert;
    p.pair_tab = pair_tab ? h->plan.pair_tab : nullptr;
    p.meta = h->plan.meta;
    p.gathered = dispatched;
    p.out = out;
    p.out_rows = static_cast<int>(rows);
    int rc;
    if ((rc = encode_2d(h, &p.tmap_a, dispatched, H, rows, static_cast<uint64_t>(H) * 2, kTileK, kTileM)) != TOVL_OK)
        return rc;
    rc = wide ? encode_weights_wide(h, &p.tmap_b, W, N, static_cast<uint64_t>(E) * H)
              : encode_weights(h, &p.tmap_b, W, N, static_cast<uint64_t>(E) * H);
    if (rc != TOVL_OK) return rc;
    if ((rc = encode_2d(h, &p.tmap_out, out, N, rows, static_cast<uint64_t>(N) * 2, kEpiBoxCols, 32,
                        CU_TENSOR_MAP_SWIZZLE_64B)) != TOVL_OK)
        return rc;
    p.seq = static_cast<int>(h->seq + 1);
    p.gate_seq = p.seq + h->fault_gate_offset;
    // (pair tiles over 128-row segments: at most one per block)
    p.trace_tiles = static_cast<int>(rows / kTileM / (pair_tab ? 1 : pair) * p.n_nb);
    if ((rc = reset_stats(h, s, p.trace_tiles, p.k_slices)) != TOVL_OK) return rc;
    e = launch(h, p, s, true, pair);
    if (e != cudaSuccess) return cuda_fail(h, e, "fused launch");
    h->seq += 1;
    h->last_stream = s;
    h->last_dispatched = dispatched;
    h->last_T = T;
    h->last_k = k;
    h->last_E = E;
    return TOVL_OK;
}

TOVL_API int tovl_gemm_reduce_scatter(tovl_handle h, const void* X, int num_shards, int M, int Ks, const void* W,
                                      int N, void* partials, void* out, void* stream)
{
    if (!h) return TOVL_ERR_INVALID;
    if (!X || !W || !partials || !out) return TOVL_ERR_INVALID;
    if (!aligned16(X) || !aligned16(W) || !aligned16(partials) || !aligned16(out)) return TOVL_ERR_INVALID;
    if (num_shards < 1 || num_shards > kMaxShards || M < 1 || Ks < kTileK || Ks % kTileK) return TOVL_ERR_INVALID;
    if (M % kTileM || Ks > kMaxK || N < kTileN || N % kTileN) return TOVL_ERR_UNSUPPORTED;
    // CTA pairs need whole 256-row tiles inside every shard
    const int pair = (h->pair_mode && h->max_pairs > 0 && (M / kTileM) % 2 == 0) ? 2 : 1;
    const int n_mb = M / kTileM;
    const int n_nb = N / kTileN;
    const long long out_tiles = static_cast<long long>(n_mb / pair) * n_nb;
    const long long tiles = out_tiles * num_shards;
    if (tiles > static_cast<long long>(h->ctrl.n_chunk_cap) * h->ctrl.n_slices) return TOVL_ERR_INVALID;
    DeviceGuard g(h->device);
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    FusedParams p;
    base_params(h, p);
    p.mode = kModeReduceScatter;
    p.M = M;
    p.N = N;
    p.K = Ks;
    p.n_kb = Ks / kTileK;
    p.n_nb = n_nb;
    p.row_bytes = N * 2;
    p.n_shards = num_shards;
    p.rows_per_shard = M;
    p.rs_tiles = static_cast<int>(tiles);
    p.rs_pair = pair;
    p.rs_join = h->role_switch ? 1 : 0;
    p.rs_out = out;
    p.out = partials;
    p.out_rows = num_shards * M;
    // reduction traffic: S partial rows read and one output row written per row
    int P, C;
    split_ctas(h, P, C, n_mb, n_nb * num_shards, 2.0 * (num_shards + 1) * M * N,
               2.0 * num_shards * static_cast<double>(M) * N * Ks, pair);
    if (h->producers == 0 && h->rs_epi) {
        // every SM (co-resident pair) computes partial tiles; the computer of
        // shard (o mod S)'s partial of output tile o sums that tile's S
        // partials in its epilogue, from L2, right after they are published
        C = (pair == 2 && 2 * h->max_pairs < h->num_sms) ? 2 * h->max_pairs : h->num_sms;
        if (h->consumers > 0 && h->consumers < C) C = h->consumers;
        if (pair == 2) C &= ~1;
        P = 0;
        h->last_P = P;
        h->last_C = C;
        p.rs_epi = 1;
        p.rs_join = 0;
    } else if (h->producers == 0 && h->role_switch) {
        // the consumers take over the reduction once their tiles are done, so
        // the producers only need to keep pace while the GEMM runs: about a
        // tenth of the SMs (measured on the TP shape: 16 of 152 best)
        P = (h->num_sms / 10 + 1) & ~1;
        if (P < 2) P = 2;
        C = h->num_sms - P;
        if (pair == 2) {
            if (C > 2 * h->max_pairs) C = 2 * h->max_pairs;
            C &= ~1;
        }
        h->last_P = P;
        h->last_C = C;
    }
    p.n_producers = P;
    p.n_consumers = C;
    p.gated = 0;
    p.k_slices = 1;
    p.item_rows = 1;
    p.wave_blocks = 1;
    int rc;
    if ((rc = encode_2d(h, &p.tmap_a, X, Ks, static_cast<uint64_t>(num_shards) * M, static_cast<uint64_t>(Ks) * 2,
                        kTileK, kTileM)) != TOVL_OK)
        return rc;
    if ((rc = encode_weights(h, &p.tmap_b, W, N, static_cast<uint64_t>(num_shards) * Ks)) != TOVL_OK) return rc;
    if ((rc = encode_2d(h, &p.tmap_out, partials, N, static_cast<uint64_t>(num_shards) * M,
                        static_cast<uint64_t>(N) * 2, kEpiBoxCols, 32, CU_TENSOR_MAP_SWIZZLE_64B)) != TOVL_OK)
        return rc;
    p.seq = static_cast<int>(h->seq + 1);
    p.gate_seq = p.seq + h->fault_gate_offset;
    p.trace_tiles = static_cast<int>(tiles);
    if ((rc = reset_stats(h, s, tiles, 1)) != TOVL_OK) return rc;
    // the reduction items of producer CTAs are handed out by a ticket
    // counter that starts at 0 (the epilogue reduction takes no tickets)
    cudaError_t e = cudaSuccess;
    if (!p.rs_epi && (e = cudaMemsetAsync(h->ctrl.work, 0, sizeof(int), s)) != cudaSuccess)
        return cuda_fail(h, e, "ticket reset");
    e = launch(h, p, s, true, pair);
    if (e != cudaSuccess) return cuda_fail(h, e, "reduce-scatter launch");
    h->seq += 1;
    h->last_stream = s;
    return TOVL_OK;
}

TOVL_API int tovl_combine(tovl_handle h, const void* y, int N, const float* gate_w, void* staging, void* combined,
                          void* stream)
{
    if (!h) return TOVL_ERR_INVALID;
    if (h->last_T <= 0 && h->last_k <= 0) return TOVL_ERR_INVALID;   // no dispatch round on this handle yet
    if (!y || !gate_w || !staging || !combined) return TOVL_ERR_INVALID;
    if (!aligned16(y) || !aligned16(staging) || !aligned16(combined) || (reinterpret_cast<uintptr_t>(gate_w) & 3u))
        return TOVL_ERR_INVALID;
    if (N < kTileK || N % kTileK) return TOVL_ERR_INVALID;
    if (N > kMaxK) return TOVL_ERR_UNSUPPORTED;
    const long long pairs = static_cast<long long>(h->last_T) * h->last_k;
    if (pairs > h->cfg.max_rows) return TOVL_ERR_INVALID;
    if (pairs == 0) return TOVL_OK;    // the last dispatch round had no tokens: nothing to combine, no round
    DeviceGuard g(h->device);
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    FusedParams p;
    base_params(h, p);
    p.mode = kModeGather;
    p.M = static_cast<int>(pairs);     // staging rows, token-major: row t*k + j
    p.N = N;
    p.K = N;
    p.n_kb = N / kTileK;
    p.n_nb = 0;
    p.row_bytes = N * 2;
    // copy traffic 2 x rows x N x 2 bytes against the reduction's k+1 rows
    // per token: 7/12 of the SMs copy, the rest reduce (measured on GB300
    // with the uniform top-2 and Zipf top-4 combines: 88 of 152 producer
    // CTAs best, 76 and 100 within 5 %, 48 and 112 25-40 % slower)
    int P = h->producers > 0 ? h->producers : h->num_sms * 7 / 12;
    if (P > h->num_sms - 1) P = h->num_sms - 1;
    p.n_producers = P;
    p.n_reducers = h->num_sms - P;
    // embedded copy (option 18, unless a producer count is set): every CTA
    // copies in its first kCombineCopyWarps warps and reduces in the others
    if (h->embedded != 0 && h->producers <= 0) {
        p.n_producers = 0;
        p.n_reducers = h->num_sms;
        p.embedded = kCombineCopyWarps;
    }
    h->last_P = p.n_producers;
    h->last_C = p.n_reducers;
    p.k_slices = 1;
    {
        const int n16 = p.n_kb * kTileK * 2 / 16;
        int ri = 64;
        while (ri > 1 && ri * n16 > kItemInt4) ri >>= 1;
        p.item_rows = ri;
    }
    p.wave_blocks = static_cast<int>(ceil_div(pairs, kBlockRows));   // one ordering group: token order
    if (p.wave_blocks < 1) p.wave_blocks = 1;
    p.x = y;
    p.src_rows = h->plan.dst;
    p.rows_valid = h->plan.meta;
    p.gate_w = gate_w;
    p.gathered = staging;
    p.combined = combined;
    p.T = h->last_T;
    p.k = h->last_k;
    p.seq = static_cast<int>(h->seq + 1);
    p.gate_seq = p.seq + h->fault_gate_offset;
    p.trace_tiles = 0;
    int rc;
    if ((rc = reset_stats(h, s, 0, 1)) != TOVL_OK) return rc;
    const bool pdl = h->pdl && h->pdl_ok;
    cudaError_t e = launch_combine(p, s, h->coop_enabled, pdl);
    if (e != cudaSuccess && (h->coop_enabled || pdl)) {
        cudaGetLastError();
        e = launch_combine(p, s, false, false);
    }
    if (e != cudaSuccess) return cuda_fail(h, e, "combine launch");
    h->seq += 1;
    h->last_stream = s;
    return TOVL_OK;
}

TOVL_API int tovl_gated_copy(tovl_handle h, const void* src, void* dst, long long n_rows, int row_bytes, const int* perm,
                             int gated, int stamps, void* stream)
{
    if (!h) return TOVL_ERR_INVALID;
    if (!src || !dst || !perm || !aligned16(src) || !aligned16(dst) || (reinterpret_cast<uintptr_t>(perm) & 3u))
        return TOVL_ERR_INVALID;
    if (n_rows < 1 || n_rows > h->cfg.max_rows || row_bytes < 16 || row_bytes % 16) return TOVL_ERR_INVALID;
    // the automatic mode: 16-byte vector copies below 8 KB rows, bulk copies
    // from 8 KB up to the largest row a bulk stage holds (measured on GB300,
    // gated, 2^20 rows: vector 4.84-6.17 TB/s from 256 B to 4 KB; bulk 6.38
    // and 6.51 TB/s at 8 and 16 KB against vector 6.17 and 6.21)
    int mode = h->copy_mode;
    if (mode == TOVL_COPY_AUTO)
        mode = (row_bytes >= kCopyAutoBulkRowBytes && row_bytes <= copy_bulk_max_row_bytes()) ? TOVL_COPY_BULK
                                                                                              : TOVL_COPY_VECTOR;
    if (mode == TOVL_COPY_BULK && row_bytes > copy_bulk_max_row_bytes()) return TOVL_ERR_UNSUPPORTED;
    DeviceGuard g(h->device);
    CopyParams p;
    std::memset(&p, 0, sizeof p);
    p.src = static_cast<const uint8_t*>(src);
    p.dst = static_cast<uint8_t*>(dst);
    p.perm = perm;
    p.n_rows = n_rows;
    p.row_bytes = row_bytes;
    p.n_chunks = static_cast<int>(ceil_div(n_rows, kChunkRows));
    p.gated = gated ? 1 : 0;
    p.timeout_ns = h->timeout_ns;
    p.pipe_timeout_ns = pipe_timeout(h);
    p.copy_mode = mode;
    p.stamps = (gated && stamps) ? 1 : 0;
    p.ctrl = h->ctrl;
    const int per_sm = copy_max_active_per_sm(p.copy_mode);
    if (per_sm < 1) return TOVL_ERR_UNSUPPORTED;
    int waiters = 0;
    if (p.gated) {
        const long long per_cta = static_cast<long long>(kCopyWarpsPerCta) * kWaiterChunksPerWarp;
        waiters = h->copy_waiters ? h->copy_waiters : static_cast<int>(ceil_div(p.n_chunks, per_cta));
        if (static_cast<long long>(waiters) * per_cta < p.n_chunks) return TOVL_ERR_INVALID;
    }
    int copiers = h->copy_ctas ? h->copy_ctas : h->num_sms * per_sm - waiters;
    if (copiers + waiters > h->num_sms * per_sm) copiers = h->num_sms * per_sm - waiters;
    if (copiers < 1) return TOVL_ERR_INVALID;
    p.n_copiers = copiers;
    p.seq = static_cast<int>(p.gated ? h->seq + 1 : h->seq);
    const cudaError_t e = launch_copy(p, waiters, h->coop_enabled, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(h, e, "copy launch");
    if (p.gated) h->seq += 1;
    h->last_stream = static_cast<cudaStream_t>(stream);
    return TOVL_OK;
}

static int sync_last(tovl_ctx* h)
{
    cudaError_t e = h->last_stream ? cudaStreamSynchronize(h->last_stream) : cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    return e == cudaSuccess ? TOVL_OK : cuda_fail(h, e, "synchronize");
}

TOVL_API int tovl_sync_status(tovl_handle h)
{
    if (!h) return TOVL_ERR_INVALID;
    DeviceGuard g(h->device);
    int rc = sync_last(h);
    if (rc != TOVL_OK) return rc;
    int st = 0;
    cudaError_t e = cudaMemcpy(&st, h->ctrl.status, sizeof st, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(h, e, "status read");
    if (st != 0) {
        e = cudaMemset(h->ctrl.status, 0, sizeof st);
        if (e != cudaSuccess) return cuda_fail(h, e, "status clear");
    }
    return st;
}

TOVL_API int tovl_ctrl_sizes(tovl_handle h, int* n_chunks, int* n_blocks)
{
    if (!h) return TOVL_ERR_INVALID;
    if (n_chunks) *n_chunks = h->ctrl.n_chunk_cap * h->ctrl.n_slices;
    if (n_blocks) *n_blocks = h->ctrl.n_block_cap * h->ctrl.n_slices;
    return TOVL_OK;
}

static int d2h(tovl_ctx* h, void* dst, const void* src, size_t bytes)
{
    if (!dst || !bytes) return TOVL_OK;
    const cudaError_t e = cudaMemcpy(dst, src, bytes, cudaMemcpyDeviceToHost);
    return e == cudaSuccess ? TOVL_OK : cuda_fail(h, e, "copy to host");
}

TOVL_API int tovl_read_ctrl(tovl_handle h, int* slots, int* cnts, int* rbcnts, long long* seq)
{
    if (!h) return TOVL_ERR_INVALID;
    DeviceGuard g(h->device);
    int rc = sync_last(h);
    const size_t nc = static_cast<size_t>(h->ctrl.n_chunk_cap) * h->ctrl.n_slices * sizeof(int);
    const size_t nb = static_cast<size_t>(h->ctrl.n_block_cap) * h->ctrl.n_slices * sizeof(int);
    if (rc == TOVL_OK) rc = d2h(h, slots, h->ctrl.slot, nc);
    if (rc == TOVL_OK) rc = d2h(h, cnts, h->ctrl.cnt, nc);
    if (rc == TOVL_OK) rc = d2h(h, rbcnts, h->ctrl.rbcnt, nb);
    if (rc == TOVL_OK && seq) *seq = h->seq;
    return rc;
}

TOVL_API int tovl_read_plan(tovl_handle h, int* counts, int* dst, int* src_of_dst, int* pad, int* blk_expert,
                            int* m_pad)
{
    if (!h) return TOVL_ERR_INVALID;
    DeviceGuard g(h->device);
    int rc = sync_last(h);
    int meta[4] = {0, 0, 0, 0};
    if (rc == TOVL_OK) rc = d2h(h, meta, h->plan.meta, sizeof meta);
    const size_t pairs = static_cast<size_t>(h->last_T) * h->last_k;
    if (rc == TOVL_OK) rc = d2h(h, counts, h->plan.counts, static_cast<size_t>(h->last_E) * sizeof(int));
    if (rc == TOVL_OK) rc = d2h(h, dst, h->plan.dst, pairs * sizeof(int));
    if (rc == TOVL_OK) rc = d2h(h, src_of_dst, h->plan.src_of_dst, static_cast<size_t>(meta[0]) * sizeof(int));
    if (rc == TOVL_OK) rc = d2h(h, pad, h->plan.pad, static_cast<size_t>(meta[1]) * sizeof(int));
    if (rc == TOVL_OK) rc = d2h(h, blk_expert, h->plan.blk_expert, static_cast<size_t>(meta[1]) * sizeof(int));
    if (rc == TOVL_OK && m_pad) *m_pad = meta[0];
    return rc;
}

TOVL_API int tovl_read_stats(tovl_handle h, unsigned long long* stats, int n)
{
    if (!h || !stats || n < 0) return TOVL_ERR_INVALID;
    DeviceGuard g(h->device);
    int rc = sync_last(h);
    if (n > kNumStats) n = kNumStats;
    if (rc == TOVL_OK) rc = d2h(h, stats, h->ctrl.stats, static_cast<size_t>(n) * sizeof(unsigned long long));
    return rc;
}

TOVL_API int tovl_read_trace(tovl_handle h, int what, long long* out, long long n)
{
    if (!h || !out || n < 0) return TOVL_ERR_INVALID;
    const long long* src = nullptr;
    long long avail = 0;
    if (what == 0) {
        src = h->ctrl.pub_ns;
        avail = static_cast<long long>(h->ctrl.n_chunk_cap) * h->ctrl.n_slices;
    } else if (what == 1) {
        src = h->ctrl.trace;
        avail = h->last_tiles * h->last_ks;
    } else if (what == 2) {
        src = h->ctrl.trace + h->last_tiles * h->last_ks;
        avail = h->last_tiles;
    } else if (what == 3) {
        src = h->ctrl.trace + h->last_tiles * (h->last_ks + 1);
        avail = h->last_tiles;
    } else {
        return TOVL_ERR_INVALID;
    }
    if (src - h->ctrl.trace >= 0 && (src - h->ctrl.trace) + avail > h->ctrl.trace_cap)
        avail = h->ctrl.trace_cap - (src - h->ctrl.trace);
    if (n > avail) return TOVL_ERR_INVALID;
    DeviceGuard g(h->device);
    int rc = sync_last(h);
    if (rc == TOVL_OK) rc = d2h(h, out, src, static_cast<size_t>(n) * sizeof(long long));
    return rc;
}

TOVL_API int tovl_read_latency(tovl_handle h, long long* pub_ns, long long* obs_ns, int n)
{
    if (!h || n < 0 || n > h->ctrl.n_chunk_cap) return TOVL_ERR_INVALID;
    DeviceGuard g(h->device);
    int rc = sync_last(h);
    if (rc == TOVL_OK) rc = d2h(h, pub_ns, h->ctrl.pub_ns, static_cast<size_t>(n) * sizeof(long long));
    if (rc == TOVL_OK) rc = d2h(h, obs_ns, h->ctrl.obs_ns, static_cast<size_t>(n) * sizeof(long long));
    return rc;
}

TOVL_API int tovl_set_option(tovl_handle h, int option, long long value)
{
    if (!h) return TOVL_ERR_INVALID;
    switch (option) {
    case 1:
        if (value < 0 || value >= h->num_sms) return TOVL_ERR_INVALID;
        h->producers = static_cast<int>(value);
        return TOVL_OK;
    case 2:
        if (value < 0 || value > h->num_sms) return TOVL_ERR_INVALID;
        h->consumers = static_cast<int>(value);
        return TOVL_OK;
    case 3:
        if (value != TOVL_COPY_VECTOR && value != TOVL_COPY_BULK && value != TOVL_COPY_AUTO) return TOVL_ERR_INVALID;
        h->copy_mode = static_cast<int>(value);
        return TOVL_OK;
    case 4:
        h->stats = value ? 1 : 0;
        return TOVL_OK;
    case 5:
        if (value < 1000) return TOVL_ERR_INVALID;
        h->timeout_ns = value;
        return TOVL_OK;
    case 6:
        if (value < 0) return TOVL_ERR_INVALID;
        h->copy_ctas = static_cast<int>(value);
        return TOVL_OK;
    case 7:
        if (value < 0) return TOVL_ERR_INVALID;
        h->copy_waiters = static_cast<int>(value);
        return TOVL_OK;
    case 8:
        if (value < 0 || value > 1000) return TOVL_ERR_INVALID;
        h->fault_gate_offset = static_cast<int>(value);
        return TOVL_OK;
    case 10:
        if (value != 0 && value != 1) return TOVL_ERR_INVALID;
        h->pair_mode = static_cast<int>(value);
        return TOVL_OK;
    case 13:
        if (value != 0 && value != 1) return TOVL_ERR_INVALID;
        h->coop_enabled = value != 0;
        return TOVL_OK;
    case 14:
        if (value != 0 && value != 1) return TOVL_ERR_INVALID;
        h->producer_mode = static_cast<int>(value);
        return TOVL_OK;
    case 15:
        if (value != 0 && value != 1) return TOVL_ERR_INVALID;
        h->pdl = value != 0;
        return TOVL_OK;
    case 16:
        if (value < 0 || value > 2) return TOVL_ERR_INVALID;
        h->role_switch = static_cast<int>(value);
        return TOVL_OK;
    case 17:
        if (value != kBlockRows && value != 2 * kBlockRows) return TOVL_ERR_INVALID;
        h->dispatch_align = static_cast<int>(value);
        return TOVL_OK;
    case 18:
        if (value < 0 || value > 2) return TOVL_ERR_INVALID;
        h->embedded = static_cast<int>(value);
        return TOVL_OK;
    case 19:
        if (value != 0 && value != 1) return TOVL_ERR_INVALID;
        h->rs_epi = static_cast<int>(value);
        return TOVL_OK;
    case 20:
        if (value < -1 || value > 63) return TOVL_ERR_INVALID;
        h->l2_hints = static_cast<int>(value);
        return TOVL_OK;
    case 23:
        if (value != 0 && value != 1) return TOVL_ERR_INVALID;
        h->wide_tiles = static_cast<int>(value);
        return TOVL_OK;
    default:
        return TOVL_ERR_INVALID;
    }
}

TOVL_API int tovl_get_option(tovl_handle h, int option, long long* value)
{
    if (!h || !value) return TOVL_ERR_INVALID;
    switch (option) {
    case 1: *value = h->last_P; return TOVL_OK;
    case 2: *value = h->last_C; return TOVL_OK;
    case 3: *value = h->copy_mode; return TOVL_OK;
    case 9: *value = h->slices; return TOVL_OK;
    case 4: *value = h->stats; return TOVL_OK;
    case 5: *value = h->timeout_ns; return TOVL_OK;
    case 6: *value = h->copy_ctas; return TOVL_OK;
    case 7: *value = h->copy_waiters; return TOVL_OK;
    case 8: *value = h->fault_gate_offset; return TOVL_OK;
    case 10: *value = (h->pair_mode && h->max_pairs > 0) ? 1 : 0; return TOVL_OK;
    case 11: *value = h->max_pairs; return TOVL_OK;
    case 12: *value = h->coop_pairs ? 1 : 0; return TOVL_OK;
    case 13: *value = h->coop_enabled ? 1 : 0; return TOVL_OK;
    case 14: *value = h->producer_mode; return TOVL_OK;
    case 15: *value = (h->pdl && h->pdl_ok) ? 1 : 0; return TOVL_OK;
    case 16: *value = h->role_switch; return TOVL_OK;
    case 17: *value = h->dispatch_align; return TOVL_OK;
    case 18: *value = h->embedded; return TOVL_OK;
    case 19: *value = h->rs_epi; return TOVL_OK;
    case 20: *value = h->l2_hints; return TOVL_OK;
    case 23: *value = h->wide_tiles; return TOVL_OK;
    default: return TOVL_ERR_INVALID;
    }
}
