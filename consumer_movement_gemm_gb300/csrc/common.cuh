// common.cuh -- helpers shared by the producer and consumer roles of the
// fused kernel.
#pragma once
#include "ctrl.cuh"
#include "ptx.cuh"

namespace tovl {

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

__device__ __forceinline__ void trace_put(const FusedParams& p, long long idx, unsigned long long v)
{
    if (p.stats && idx < p.ctrl.trace_cap) p.ctrl.trace[idx] = static_cast<long long>(v);
}

// L2 cache policy of one stream: `last_bit` set -> evict last, `first_bit`
// set -> evict first, neither -> evict normal (bits of FusedParams::l2_hints).
__device__ __forceinline__ uint64_t stream_policy(const FusedParams& p, int last_bit, int first_bit)
{
    return ptx::l2_policy((p.l2_hints & last_bit) ? 2 : (p.l2_hints & first_bit) ? 1 : 0);
}

// Number of 128-row blocks the producers fill and the consumers traverse.
// Rows of a gather-mode round: p.M, or none when the round's row table comes
// from a routing plan that was rejected.
__device__ __forceinline__ int gather_rows(const FusedParams& p)
{
    return (p.rows_valid && p.rows_valid[1] <= 0) ? 0 : p.M;
}

// Row blocks of a round (for reduce-scatter: of one shard).
__device__ __forceinline__ int num_row_blocks(const FusedParams& p)
{
    if (p.mode == kModeGather) return (gather_rows(p) + kTileM - 1) / kTileM;
    if (p.mode == kModeReduceScatter) return p.M / kTileM;
    return p.meta[1];
}

// K-blocks [kb_begin(s), kb_begin(s+1)) form slice s.
__device__ __forceinline__ int kb_begin(const FusedParams& p, int s)
{
    return s * p.n_kb / p.k_slices;
}

}  // namespace tovl
