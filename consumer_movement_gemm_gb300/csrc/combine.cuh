// combine.cuh -- reducer CTAs of the combine kernel.
//
// Combine is dispatch in reverse ("cross-GPU sync protocols on PCIe",
// section 3: the layer-1 combine pushes each expert-output row back to its
// token's staging row and the last writer of a chunk, elected by an acq_rel
// count, publishes the chunk's slot).  The producer CTAs of the combine
// kernel are the fused kernel's producers with a row table: staging row
// t*k + j copies expert-output row dst(t, j).  The reducers below wait for
// the slots of the chunks that hold a token's k staged rows (acquire polls
// of local slots, warp vote) and write the token's combined row
//   combined[t, :] = bf16( sum_j w[t*k + j] * staging[t*k + j, :] ),
// every product and every partial sum rounded to fp32, j ascending.
#pragma once
#include "common.cuh"
#include "ctrl.cuh"
#include "ptx.cuh"
#include "sync.cuh"

namespace tovl {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// The weighted sum of token t's k staged rows.  A lane's column groups are
// lane, lane + 32, ... below N / 8; kBatch of them from KR staged rows are
// loaded together (up to 16 loads in flight per lane), so a token with k <= 4
// costs one round trip per batch (a group past the row loads the lane's
// first one again and is not stored; with k > 4, a row past k in the last
// batch of rows re-reads the token's last row, whose product is skipped).
template <int KR>
__device__ __forceinline__ void combine_token(const FusedParams& p, int t, int lane, const uint8_t* staging, uint8_t* out,
                                              int groups, size_t row_bytes)
{
    constexpr int kBatch = 4;
    const int s0 = t * p.k;
    const int per_lane = (groups + 31) / 32;
    for (int i0 = 0; i0 < per_lane; i0 += kBatch) {
        float acc[kBatch][8];
#pragma unroll
        for (int b = 0; b < kBatch; ++b)
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[b][c] = 0.0f;
        for (int j0 = 0; j0 < p.k; j0 += KR) {
            float w[KR];
            int4 v[KR][kBatch];
#pragma unroll
            for (int jj = 0; jj < KR; ++jj) {
                const int j = min(j0 + jj, p.k - 1);
                w[jj] = p.gate_w[s0 + j];
                const int4* row = reinterpret_cast<const int4*>(staging + static_cast<size_t>(s0 + j) * row_bytes);
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                    const int g = lane + 32 * (i0 + b);
                    v[jj][b] = ptx::ld_v4(row + (g < groups ? g : lane % groups));
                }
            }
            // products and sums in ascending j
#pragma unroll
            for (int jj = 0; jj < KR; ++jj) {
                if (j0 + jj >= p.k) break;
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                    const uint32_t u[4] = {static_cast<uint32_t>(v[jj][b].x), static_cast<uint32_t>(v[jj][b].y),
                                           static_cast<uint32_t>(v[jj][b].z), static_cast<uint32_t>(v[jj][b].w)};
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        acc[b][2 * c] = __fadd_rn(acc[b][2 * c], __fmul_rn(w[jj], bf16_lo(u[c])));
                        acc[b][2 * c + 1] = __fadd_rn(acc[b][2 * c + 1], __fmul_rn(w[jj], bf16_hi(u[c])));
                    }
                }
            }
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int g = lane + 32 * (i0 + b);
            if (g >= groups) break;
            int4 o;
            o.x = static_cast<int>(ptx::pack_bf16x2(acc[b][0], acc[b][1]));
            o.y = static_cast<int>(ptx::pack_bf16x2(acc[b][2], acc[b][3]));
            o.z = static_cast<int>(ptx::pack_bf16x2(acc[b][4], acc[b][5]));
            o.w = static_cast<int>(ptx::pack_bf16x2(acc[b][6], acc[b][7]));
            ptx::st_v4(reinterpret_cast<int4*>(out + static_cast<size_t>(t) * row_bytes) + g, o);
        }
    }
}

// Reducer warps first_warp .. 15 of reducer unit `rid` of `n_units` (a
// reducer CTA, or every CTA when the copy runs in its other warps).
__device__ inline void reducer(const FusedParams& p, int rid, int n_units, int first_warp)
{
    const int warp = threadIdx.x / 32;
    const int lane = static_cast<int>(ptx::lane_id());
    if (gather_rows(p) == 0) {
        // the routing plan of the round was rejected: nothing to combine
        if (rid == 0 && warp == first_warp && lane == 0) record_error(p.ctrl, kErrInvalid);
        return;
    }
    // consecutive tokens go to different CTAs, in the producers' order
    const int gw = (warp - first_warp) * n_units + rid;
    const int n_gw = n_units * (kThreads / 32 - first_warp);
    const int S = p.ctrl.n_slices;
    const int groups = p.N / 8;   // 16-byte column groups of a row
    const size_t row_bytes = static_cast<size_t>(p.N) * 2;
    const uint8_t* staging = static_cast<const uint8_t*>(p.gathered);
    uint8_t* out = static_cast<uint8_t*>(p.combined);
    for (int t = gw; t < p.T; t += n_gw) {
        const int s0 = t * p.k;
        // every chunk that holds one of the token's k staged rows: one or two
        // for k <= 65, more for larger k (lane i watches chunk c0 + i, 32
        // chunks per pass)
        const int c0 = s0 / kChunkRows, c1 = (s0 + p.k - 1) / kChunkRows;
        for (int cb = c0; cb <= c1; cb += 32) {
            const int c = cb + lane;
            if (warp_wait_lanes(c <= c1 ? p.ctrl.slot + c * S : nullptr, p.gate_seq, p.ctrl, p.seq,
                                p.timeout_ns) < 0)
                return;
        }
        // the token's weighted sum, min(k, 4) staged rows' loads in flight together
        if (p.k >= 4) combine_token<4>(p, t, lane, staging, out, groups, row_bytes);
        else if (p.k == 3) combine_token<3>(p, t, lane, staging, out, groups, row_bytes);
        else if (p.k == 2) combine_token<2>(p, t, lane, staging, out, groups, row_bytes);
        else combine_token<1>(p, t, lane, staging, out, groups, row_bytes);
    }
}

}  // namespace tovl
