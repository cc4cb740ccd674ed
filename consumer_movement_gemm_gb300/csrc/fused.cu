// fused.cu -- the persistent fused gather/dispatch + GEMM kernel.
//
// One cooperative launch of P producer CTAs and C consumer CTAs, one CTA per
// SM, all co-resident:
//   producers  copy token rows into the gathered (or dispatched) buffer and
//              count them with the single-writer protocol: 64-row chunk
//              watermarks published by an elected last arrival (gather), or
//              release reductions into 128-row block counters pre-seeded
//              with the padding count (dispatch)  -- "cross-GPU sync
//              protocols on PCIe", sections 3-5;
//   consumers  run a tcgen05 bf16 GEMM over 128x256 output tiles in
//              row-block order (the producers' order, section 6 item 3); the
//              TMA warp of each consumer gates every new row block on the
//              protocol with acquire polls before loading it.
// Producers never wait on anyone; consumers wait only on producers, which are
// resident by construction (cooperative launch), and every wait is bounded.
#include <cuda_runtime.h>
#include "ctrl.cuh"
#include "ptx.cuh"
#include "sync.cuh"
#include "copyplane.cuh"
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

// Number of 128-row blocks the consumers traverse.
__device__ __forceinline__ int num_row_blocks(const FusedParams& p)
{
    if (p.mode == kModeGather) return (p.M + kTileM - 1) / kTileM;
    return p.meta[1];
}

// Rows of the gathered/dispatched buffer the producers fill this round.
__device__ __forceinline__ int num_rows(const FusedParams& p)
{
    if (p.mode == kModeGather) return p.M;
    return p.meta[0];
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
    return s;
}

// TMA warp: gate each new row block, then stream A and B k-blocks.
__device__ void consumer_tma(const FusedParams& p, const ConsumerSmem& s, int cid, int n_tiles)
{
    const uint32_t lane = ptx::lane_id();
    uint32_t stage = 0, phase = 0;
    int gated_mb = -1;
    unsigned long long polls = 0;
    for (int t = cid; t < n_tiles; t += p.n_consumers) {
        const int mb = t / p.n_nb;
        const int nb = t % p.n_nb;
        int brow = 0;
        if (p.mode == kModeDispatch) brow = p.blk_expert[mb] * p.K;
        if (p.gated && mb != gated_mb) {
            const int* words[2];
            int n = 0;
            int target;
            if (p.mode == kModeGather) {
                const int c0 = mb * (kTileM / kChunkRows);
                for (int i = 0; i < kTileM / kChunkRows; ++i)
                    if ((c0 + i) * kChunkRows < p.M) words[n++] = p.ctrl.slot + c0 + i;
                target = p.gate_seq;
            } else {
                words[n++] = p.ctrl.rbcnt + mb;
                target = p.gate_seq * kBlockRows;
            }
            const int r = warp_wait_ge(words, n, target, p.ctrl, p.seq, p.timeout_ns);
            polls += static_cast<unsigned long long>(r < 0 ? -r : r);
            gated_mb = mb;
            // the gathered rows were written through the generic proxy (or
            // bulk copies); order them before this thread's TMA reads.
            if (lane == 0) ptx::fence_proxy_async_global();
        }
        int fail = 0;
        if (lane == 0) {
            for (int kb = 0; kb < p.n_kb; ++kb) {
                if (!mbar_wait(&s.empty[stage], phase ^ 1u, p.ctrl, p.pipe_timeout_ns)) {
                    fail = 1;
                    break;
                }
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
        if (__shfl_sync(0xffffffffu, fail, 0)) break;
    }
    if (p.stats && lane == 0 && polls) atomicAdd(p.ctrl.stats + kStatGatePolls, polls);
}

// MMA warp: one elected lane issues tcgen05.mma into a double-buffered TMEM
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
__device__ void consumer_epilogue(const FusedParams& p, const ConsumerSmem& s, int cid, int n_tiles,
                                  uint32_t tmem_base, int valid_rows)
{
    const int warp = threadIdx.x / 32;
    const uint32_t lane = ptx::lane_id();
    const int q = warp & 3;                       // TMEM lane quarter this warp may access
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
        uint4* dst = reinterpret_cast<uint4*>(out + static_cast<size_t>(row) * p.N + nb * kTileN);
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kTileN;
#pragma unroll 1
        for (int c = 0; c < kTileN / 32; ++c) {
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
            ptx::mbar_init(&s.tempty[i], 4 * 32);
        }
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
    else consumer_epilogue(p, s, cid, n_tiles, tmem_base, valid_rows);
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
// Completion of one copied row.
__device__ __forceinline__ void row_done(const FusedParams& p, int r)
{
    if (p.mode == kModeGather) {
        arrive_and_publish(p.ctrl, r / kChunkRows, 1, p.seq);
    } else {
        ptx::red_add_release_gpu(p.ctrl.rbcnt + r / kBlockRows, 1);
    }
}

__device__ __forceinline__ const uint8_t* row_src(const FusedParams& p, int r)
{
    if (p.mode == kModeGather) {
        const int s = r / p.rows_per_shard;
        const int i = r - s * p.rows_per_shard;
        return static_cast<const uint8_t*>(p.shard[s]) + static_cast<size_t>(i) * p.row_bytes;
    }
    return static_cast<const uint8_t*>(p.x) + static_cast<size_t>(p.src_of_dst[r]) * p.row_bytes;
}

__device__ __forceinline__ bool row_real(const FusedParams& p, int r)
{
    return p.mode == kModeGather || p.src_of_dst[r] >= 0;
}

// Per-round padding seeds.  Each counter must gain exactly its per-round
// quota (64 per chunk, 128 per row block) every call, so counters this call
// does not fill receive the missing arrivals as one seed add.
__device__ void seed_counters(const FusedParams& p, int gw, int n_gw)
{
    const uint32_t lane = ptx::lane_id();
    const Ctrl& c = p.ctrl;
    // chunk counters
    for (int ch = gw * 32 + lane; ch < c.n_chunk_cap; ch += n_gw * 32) {
        int seed = kChunkRows;
        if (p.mode == kModeGather) {
            const int real = min(max(p.M - ch * kChunkRows, 0), kChunkRows);
            seed = kChunkRows - real;
        }
        if (seed > 0) arrive_and_publish(c, ch, seed, p.seq);
    }
    // row-block counters
    if (p.mode == kModeGather) {
        for (int b = gw * 32 + lane; b < c.n_block_cap; b += n_gw * 32) ptx::red_add_release_gpu(c.rbcnt + b, kBlockRows);
        return;
    }
    const int n_blocks = p.meta[1];
    const int zero = p.meta[2];
    for (int b = gw; b < c.n_block_cap; b += n_gw) {
        if (b >= n_blocks) {
            if (lane == 0) ptx::red_add_release_gpu(c.rbcnt + b, kBlockRows);
            continue;
        }
        const int pad = p.pad[b];
        if (pad == 0) continue;
        if (zero) {
            // padding rows are the last `pad` rows of the block; they must be
            // zero before the counter reaches its target
            uint8_t* base = static_cast<uint8_t*>(p.gathered) +
                            static_cast<size_t>(b * kBlockRows + kBlockRows - pad) * p.row_bytes;
            int4* d = reinterpret_cast<int4*>(base);
            const size_t n16 = static_cast<size_t>(pad) * p.row_bytes / 16;
            const int4 z = make_int4(0, 0, 0, 0);
            for (size_t i = lane; i < n16; i += 32) ptx::st_v4(d + i, z);
            __syncwarp();
        }
        if (lane == 0) ptx::red_add_release_gpu(c.rbcnt + b, pad);
    }
}

// 16-byte vector copy, one warp per row.
__device__ void producer_v4(const FusedParams& p, int gw, int n_gw)
{
    const uint32_t lane = ptx::lane_id();
    const int rows = num_rows(p);
    const int n16 = p.row_bytes / 16;
    for (int r = gw; r < rows; r += n_gw) {
        if (!row_real(p, r)) continue;
        const int4* s = reinterpret_cast<const int4*>(row_src(p, r));
        int4* d = reinterpret_cast<int4*>(static_cast<uint8_t*>(p.gathered) + static_cast<size_t>(r) * p.row_bytes);
        int i = lane;
        for (; i + 96 < n16; i += 128) {
            const int4 v0 = ptx::ld_nc_v4(s + i);
            const int4 v1 = ptx::ld_nc_v4(s + i + 32);
            const int4 v2 = ptx::ld_nc_v4(s + i + 64);
            const int4 v3 = ptx::ld_nc_v4(s + i + 96);
            ptx::st_v4(d + i, v0);
            ptx::st_v4(d + i + 32, v1);
            ptx::st_v4(d + i + 64, v2);
            ptx::st_v4(d + i + 96, v3);
        }
        for (; i < n16; i += 32) ptx::st_v4(d + i, ptx::ld_nc_v4(s + i));
        __syncwarp();
        if (lane == 0) row_done(p, r);
    }
}

// Rows this issuer moves with bulk copies: rows g, g + n_g, ... (real rows only).
struct FusedRowJob {
    const FusedParams* p;
    int cursor;
    int step;
    int rows;
    __device__ int next()
    {
        while (cursor < rows) {
            const int r = cursor;
            cursor += step;
            if (row_real(*p, r)) return r;
        }
        return -1;
    }
    __device__ const void* src(int r) { return row_src(*p, r); }
    __device__ void* dst(int r)
    {
        return static_cast<uint8_t*>(p->gathered) + static_cast<size_t>(r) * p->row_bytes;
    }
    __device__ void done(int r) { row_done(*p, r); }
};

__device__ void producer(const FusedParams& p, uint8_t* smem, int pid)
{
    const int warp = threadIdx.x / 32;
    const int n_warps = kThreads / 32;
    if (threadIdx.x == 0) stat_min(p, kStatProdStartNs, ptx::globaltimer());
    if (p.copy_mode == 0) {
        seed_counters(p, pid * n_warps + warp, p.n_producers * n_warps);
        producer_v4(p, pid * n_warps + warp, p.n_producers * n_warps);
    } else {
        if (warp == 0) {
            if (ptx::lane_id() == 0) {
                FusedRowJob job{&p, pid, p.n_producers, num_rows(p)};
                const Ring ring = make_ring(smem, kStages * kStageBytes, p.row_bytes);
                run_bulk(job, static_cast<uint32_t>(p.row_bytes), ring, p.ctrl, p.pipe_timeout_ns);
            }
            __syncwarp();
        } else {
            seed_counters(p, pid * (n_warps - 1) + warp - 1, p.n_producers * (n_warps - 1));
        }
    }
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

}  // namespace tovl

namespace tovl {

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
