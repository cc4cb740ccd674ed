// plan.cu -- routing plan for dispatch rounds.
//
// The notify stage of the DeepEP FIFO-pipeline page counts tokens per expert
// before the data moves; here the count also fixes every destination row.
// Rows of one expert are laid out in ascending (token, k) order, so the
// dispatched buffer depends on the routing alone (atomic slot claims would
// make the order, and hence the buffer, nondeterministic).  Each expert's
// segment is padded to a multiple of 128 rows; the padding count of a block
// is the seed its arrival counter receives ("cross-GPU sync protocols on
// PCIe", section 5).
//
//   plan_count     one CTA per 1024 routed pairs: per-warp match_any ranks,
//                  per-segment per-expert counts and in-segment ranks
//   plan_finalize  one CTA: per-expert prefix over segments, padded offsets,
//                  block -> expert / padding tables, destination rows and the
//                  inverse map (token of each destination row)
#include <cuda_runtime.h>
#include "ctrl.cuh"
#include "ptx.cuh"
#include "launch.cuh"

namespace tovl {

constexpr int kPlanThreads = 1024;
constexpr int kPlanWarps = kPlanThreads / 32;


__global__ void __launch_bounds__(kPlanThreads) plan_count_kernel(const PlanParams p)
{
    extern __shared__ int wcnt[];               // [kPlanWarps][E]
    ptx::grid_dep_launch();                     // the finalize kernel may start its launch
    const int tid = threadIdx.x;
    const int warp = tid / 32;
    const int lane = tid % 32;
    for (int i = tid; i < kPlanWarps * p.E; i += kPlanThreads) wcnt[i] = 0;
    __syncthreads();
    const int i = blockIdx.x * kPlanThreads + tid;
    int e = -1;
    if (i < p.n_pairs) {
        e = p.topk[i];
        if (e < 0 || e >= p.E) {
            ptx::atom_cas_relaxed_gpu(p.status, kOk, kErrInvalid);
            p.plan.meta[3] = 1;
            e = -1;
        }
    }
    // lanes routed to the same expert; rank = earlier lanes with that expert
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int rank_in_warp = __popc(same & ((1u << lane) - 1u));
    if (e >= 0 && rank_in_warp == 0) wcnt[warp * p.E + e] = __popc(same);
    __syncthreads();
    // exclusive scan over warps, per expert; segment totals to global
    for (int x = tid; x < p.E; x += kPlanThreads) {
        int run = 0;
        for (int w = 0; w < kPlanWarps; ++w) {
            const int v = wcnt[w * p.E + x];
            wcnt[w * p.E + x] = run;
            run += v;
        }
        p.plan.seg_count[blockIdx.x * p.E + x] = run;
    }
    __syncthreads();
    if (i < p.n_pairs) p.plan.local_rank[i] = (e >= 0) ? wcnt[warp * p.E + e] + rank_in_warp : 0;
}

// Expert of padded row r: the last e with off[e] <= r (empty experts share
// their start with the next one).  off[E] is past every row.
__device__ __forceinline__ int expert_of_row(const int* s_off, int E, int r)
{
    int lo = 0, hi = E;             // invariant: s_off[lo] <= r < s_off[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_off[mid] <= r) lo = mid;
        else hi = mid;
    }
    return lo;
}

// Segment bases of the finalize kernel live in shared memory when they fit
// (the destination step then needs one round of global loads, not two).
constexpr int kSegSmemInts = 10 * 1024;   // with E <= 512 the kernel stays under 48 KB

// One CTA.  Every step issues its global loads together before it uses them
// (a single thread walking dependent loads would pay one L2 round trip per
// element), and the table writes of the last step need no barrier between
// them.
__global__ void __launch_bounds__(kPlanThreads) plan_finalize_kernel(const PlanParams p)
{
    extern __shared__ int sm[];
    int* s_off = sm;                // [E+1]
    int* s_cnt = sm + p.E + 1;      // [E]
    int* s_seg = sm + 2 * p.E + 1;  // [n_seg][E] segment bases, when they fit
    const bool seg_in_smem = p.n_seg * p.E <= kSegSmemInts;
    int* s_pb = s_seg + (seg_in_smem ? p.n_seg * p.E : 0);   // [E+1] first pair tile of each segment
    int* seg_base = seg_in_smem ? s_seg : p.plan.seg_count;
    __shared__ int s_zero;
    __shared__ int s_bad;
    // the counting grid (launched just before, programmatically) has finished
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();         // the fused kernel may start its launch and prologue
    const int tid = threadIdx.x;
    if (tid == 0 && p.work) *p.work = 0;   // the fused kernel's tile tickets start at 0
    if (tid == 0) {
        s_zero = p.force_zero;
        s_bad = p.plan.meta[3];
    }
    // The routing and in-segment ranks of this thread's first kDstBatch pairs
    // do not depend on the prefix below: their loads go out with it.
    constexpr int kDstBatch = 8;
    int e0[kDstBatch], lr0[kDstBatch];
#pragma unroll
    for (int j = 0; j < kDstBatch; ++j) {
        const int i = j * kPlanThreads + tid;
        e0[j] = i < p.n_pairs ? p.topk[i] : 0;
        lr0[j] = i < p.n_pairs ? p.plan.local_rank[i] : 0;
    }
    // per-expert prefix over segments (each segment's base rank), segments
    // read kPrefixBatch at a time; the previous layout is read alongside
    constexpr int kPrefixBatch = 8;
    int prev = 0;
    if (tid <= p.E) prev = p.plan.prev_off[tid];
    for (int e = tid; e < p.E; e += kPlanThreads) {
        int run = 0;
        for (int s0 = 0; s0 < p.n_seg; s0 += kPrefixBatch) {
            int v[kPrefixBatch];
#pragma unroll
            for (int j = 0; j < kPrefixBatch; ++j)
                v[j] = (s0 + j < p.n_seg) ? p.plan.seg_count[(s0 + j) * p.E + e] : 0;
#pragma unroll
            for (int j = 0; j < kPrefixBatch; ++j) {
                if (s0 + j < p.n_seg) seg_base[(s0 + j) * p.E + e] = run;
                run += v[j];
            }
        }
        s_cnt[e] = run;
        p.plan.counts[e] = run;
    }
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        s_off[0] = 0;
        for (int e = 0; e < p.E; ++e) {
            run += (s_cnt[e] + p.align - 1) / p.align * p.align;
            s_off[e + 1] = run;
        }
        if (run > p.row_cap || run / kBlockRows > p.block_cap) s_bad = 1;
        // pair tiles: ceil(blocks / 2) per segment
        int pb = 0;
        for (int e = 0; e < p.E; ++e) {
            s_pb[e] = pb;
            pb += ((s_off[e + 1] - s_off[e]) / kBlockRows + 1) / 2;
        }
        s_pb[p.E] = pb;
    }
    __syncthreads();
    if (tid <= p.E && prev != s_off[tid]) s_zero = 1;     // benign race: every writer stores 1
    for (int e = tid + kPlanThreads; e <= p.E; e += kPlanThreads)
        if (p.plan.prev_off[e] != s_off[e]) s_zero = 1;
    __syncthreads();
    if (s_bad != 0) {
        if (tid == 0) {
            ptx::atom_cas_relaxed_gpu(p.status, kOk, kErrInvalid);
            p.plan.meta[0] = 0;
            p.plan.meta[1] = 0;
            p.plan.meta[2] = 0;
            p.plan.meta[3] = 0;
            if (p.plan.pair_tab) p.plan.pair_tab[0] = 0;
        }
        for (int e = tid; e <= p.E; e += kPlanThreads) p.expert_offsets[e] = 0;
        return;
    }
    for (int e = tid; e <= p.E; e += kPlanThreads) {
        p.plan.off[e] = s_off[e];
        p.plan.prev_off[e] = s_off[e];
        p.expert_offsets[e] = s_off[e];
    }
    const int m_pad = s_off[p.E];
    if (tid == 0) {
        p.plan.meta[0] = m_pad;
        p.plan.meta[1] = m_pad / kBlockRows;
        p.plan.meta[2] = s_zero;
        p.plan.meta[3] = 0;
        if (p.plan.pair_tab) p.plan.pair_tab[0] = s_pb[p.E];
    }
    // destination row of every pair and the inverse map, kDstBatch pairs per
    // thread at a time: the routing and in-segment ranks are loaded together
    // (the first batch's were loaded at the start)
    for (int i0 = 0; i0 < p.n_pairs; i0 += kPlanThreads * kDstBatch) {
        int e[kDstBatch], lr[kDstBatch];
#pragma unroll
        for (int j = 0; j < kDstBatch; ++j) {
            const int i = i0 + j * kPlanThreads + tid;
            e[j] = i0 == 0 ? e0[j] : (i < p.n_pairs ? p.topk[i] : 0);
            lr[j] = i0 == 0 ? lr0[j] : (i < p.n_pairs ? p.plan.local_rank[i] : 0);
        }
#pragma unroll
        for (int j = 0; j < kDstBatch; ++j) {
            const int i = i0 + j * kPlanThreads + tid;
            if (i < p.n_pairs) {
                const int d = s_off[e[j]] + seg_base[(i / kPlanThreads) * p.E + e[j]] + lr[j];
                p.plan.dst[i] = d;
                p.plan.src_of_dst[d] = i / p.k;
            }
        }
    }
    // block tables: a block holds min(128, rows of its segment left) real
    // rows, the rest is padding (with 256-row segments the last two blocks
    // of a segment may both be padded)
    for (int b = tid; b < m_pad / kBlockRows; b += kPlanThreads) {
        const int e = expert_of_row(s_off, p.E, b * kBlockRows);
        p.plan.blk_expert[b] = e;
        const int real = min(max(s_cnt[e] - (b * kBlockRows - s_off[e]), 0), kBlockRows);
        p.plan.pad[b] = kBlockRows - real;
        const int rel = b - s_off[e] / kBlockRows;
        if (p.plan.pair_tab && (rel & 1) == 0)
            p.plan.pair_tab[1 + s_pb[e] + rel / 2] = 2 * b + ((b + 1) * kBlockRows < s_off[e + 1] ? 1 : 0);
    }
    // padding rows (fewer than `align` per expert) have no source token
    for (int x = tid; x < p.E * p.align; x += kPlanThreads) {
        const int e = x / p.align;
        const int r = s_off[e] + s_cnt[e] + x % p.align;
        if (r < s_off[e + 1]) p.plan.src_of_dst[r] = -1;
    }
}

}  // namespace tovl

namespace tovl {

// The finalize kernel is launched with a programmatic edge on the counting
// grid when `pdl` is set (it waits for the counts with griddepcontrol.wait).
cudaError_t launch_plan(const PlanParams& p, cudaStream_t stream, bool pdl)
{
    const size_t sm_count = static_cast<size_t>(kPlanWarps) * p.E * sizeof(int);
    const size_t seg = static_cast<size_t>(p.n_seg) * p.E;
    const size_t sm_fin = (3 * static_cast<size_t>(p.E) + 2 + (seg <= kSegSmemInts ? seg : 0)) * sizeof(int);
    if (p.n_seg > 0) {
        plan_count_kernel<<<p.n_seg, kPlanThreads, sm_count, stream>>>(p);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(1);
    lc.blockDim = dim3(kPlanThreads);
    lc.dynamicSmemBytes = sm_fin;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = (pdl && p.n_seg > 0) ? 1 : 0;
    return cudaLaunchKernelEx(&lc, plan_finalize_kernel, p);
}

cudaError_t prepare_plan()
{
    return cudaFuncSetAttribute(plan_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kPlanWarps * kMaxExperts * static_cast<int>(sizeof(int)));
}

}  // namespace tovl
