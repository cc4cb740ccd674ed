// plan_static.cu -- the routing plan for callers that cannot allocate.
//
// tovl_dispatch_plan_noalloc runs the same two plan kernels as a dispatch
// call (plan.cu), but every scratch array they need lives in one file-scope
// device array below instead of in a handle's cudaMalloc'ed plan scratch.
// It exists for callers that must not allocate device memory themselves:
// code running inside another framework's memory budget, latency-critical
// loops that cannot afford cudaMalloc's device-wide synchronisation, and
// plugins whose host application owns every allocation.  The caller still
// passes the routing in and the two outputs out.
//
// The array is a plain static __device__ object: every GPU that loads the
// library holds it (about 0.3 MB) until the process exits, and all calls on
// a device share it, so calls whose kernels overlap on that GPU race on it.
#include <cuda_runtime.h>
#include <cstddef>
#include <mutex>

#include "tovl.h"
#include "ctrl.cuh"
#include "launch.cuh"

#define TOVL_API extern "C" __attribute__((visibility("default")))

namespace tovl {
namespace {

constexpr int kNaPairs = TOVL_NOALLOC_MAX_PAIRS;
constexpr int kNaExperts = TOVL_NOALLOC_MAX_EXPERTS;
constexpr int kNaSegs = (kNaPairs + 1023) / 1024;                                  // one per 1024 pairs
constexpr int kNaRows = (kNaPairs + kNaExperts * (kBlockRows - 1) + kBlockRows - 1) / kBlockRows * kBlockRows;
constexpr int kNaBlocks = kNaRows / kBlockRows;

// Word offsets of each scratch piece inside the array (each 64-word aligned).
constexpr size_t align64(size_t x) { return (x + 63) & ~static_cast<size_t>(63); }
constexpr size_t kOffCounts = 0;
constexpr size_t kOffOff = align64(kOffCounts + kNaExperts);
constexpr size_t kOffPrev = align64(kOffOff + kNaExperts + 1);
constexpr size_t kOffSeg = align64(kOffPrev + kNaExperts + 1);
constexpr size_t kOffRank = align64(kOffSeg + static_cast<size_t>(kNaSegs) * kNaExperts);
constexpr size_t kOffSrc = align64(kOffRank + kNaPairs);
constexpr size_t kOffPad = align64(kOffSrc + kNaRows);
constexpr size_t kOffBlk = align64(kOffPad + kNaBlocks);
constexpr size_t kOffMeta = align64(kOffBlk + kNaBlocks);
constexpr size_t kOffStatus = align64(kOffMeta + 4);
constexpr size_t kScratchWords = align64(kOffStatus + 1);

static __device__ __align__(256) int g_plan_scratch[kScratchWords];

// Host-side address of g_plan_scratch per device, looked up once per device.
std::mutex g_lock;
int* g_scratch_addr[64] = {};

}  // namespace
}  // namespace tovl

TOVL_API int tovl_dispatch_plan_noalloc(const int* topk_idx, int T, int k, int E, int* expert_offsets, int* dst_rows,
                                        void* stream)
{
    using namespace tovl;
    if (!topk_idx || !expert_offsets || !dst_rows) return TOVL_ERR_INVALID;
    if (T < 0 || k < 1 || E < 1) return TOVL_ERR_INVALID;
    const long long pairs = static_cast<long long>(T) * k;
    // sizes beyond the fixed scratch are refused before anything is enqueued
    if (pairs > kNaPairs || E > kNaExperts) return TOVL_ERR_UNSUPPORTED;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TOVL_ERR_CUDA;
    int* base = nullptr;
    {
        // One-time set-up per device, with that device current: the host
        // name g_plan_scratch is only a stand-in, so ask the runtime for the
        // array's device address.  The first call on a device does this.
        std::lock_guard<std::mutex> guard(g_lock);
        if (!g_scratch_addr[dev]) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_plan_scratch) != cudaSuccess || !p) {
                cudaGetLastError();
                return TOVL_ERR_CUDA;
            }
            g_scratch_addr[dev] = static_cast<int*>(p);
        }
        base = g_scratch_addr[dev];
    }
    const cudaStream_t s = static_cast<cudaStream_t>(stream);

    PlanParams pp{};
    pp.topk = topk_idx;
    pp.n_pairs = static_cast<int>(pairs);
    pp.k = k;
    pp.E = E;
    pp.n_seg = static_cast<int>((pairs + 1023) / 1024);
    pp.row_cap = kNaRows;
    pp.block_cap = kNaBlocks;
    pp.force_zero = 0;
    pp.expert_offsets = expert_offsets;
    pp.plan.counts = base + kOffCounts;
    pp.plan.off = base + kOffOff;
    pp.plan.prev_off = base + kOffPrev;
    pp.plan.seg_count = base + kOffSeg;
    pp.plan.local_rank = base + kOffRank;
    pp.plan.dst = dst_rows;
    pp.plan.src_of_dst = base + kOffSrc;
    pp.plan.pad = base + kOffPad;
    pp.plan.blk_expert = base + kOffBlk;
    pp.plan.meta = base + kOffMeta;
    pp.status = base + kOffStatus;
    pp.align = kBlockRows;
    // The array keeps the previous call's contents; the routing-error flag in
    // meta must start at zero (every other piece is overwritten before use).
    if (cudaMemsetAsync(base + kOffMeta, 0, 4 * sizeof(int), s) != cudaSuccess) return TOVL_ERR_CUDA;
    return launch_plan(pp, s, false) == cudaSuccess ? TOVL_OK : TOVL_ERR_CUDA;
}
