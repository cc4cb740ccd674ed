// launch.cuh -- internal launchers (one per kernel translation unit).
#pragma once
#include <cuda_runtime.h>
#include "ctrl.cuh"

namespace tovl {

cudaError_t launch_fused(const FusedParams& p, cudaStream_t stream, bool cooperative, int pair, bool pdl);
cudaError_t prepare_fused();
int fused_max_active_per_sm();
int fused_max_active_pairs();

// Combine with embedded copies: copy warps per CTA (the other warps reduce).
// Measured on GB300 against 88 producer CTAs and 64 reducer CTAs: uniform
// top-2 26.6 -> 24.7 us, Zipf top-4 72.3 -> 67.4 us; 6, 8, 11, 12 and 13 copy
// warps slower; 9 trades 1 us on the uniform combine for 1.6 us on the Zipf.
constexpr int kCombineCopyWarps = 10;
cudaError_t launch_combine(const FusedParams& p, cudaStream_t stream, bool cooperative, bool pdl);
cudaError_t prepare_combine();

cudaError_t launch_plan(const PlanParams& p, cudaStream_t stream, bool pdl);
cudaError_t prepare_plan();

cudaError_t launch_copy(const CopyParams& p, int n_waiters, bool cooperative, cudaStream_t stream);
cudaError_t prepare_copy();
int copy_max_active_per_sm(int copy_mode);
int copy_bulk_max_row_bytes();
constexpr int kCopyWarpsPerCta = 16;
constexpr int kCopyAutoBulkRowBytes = 8192;    // TOVL_COPY_AUTO takes bulk copies from this row size
constexpr int kWaiterChunksPerWarp = 8 * 32;   // one pass of eight slots per lane

}  // namespace tovl
