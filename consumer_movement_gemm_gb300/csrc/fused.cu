// fused.cu -- the persistent fused gather/dispatch + GEMM kernel.
//
// One launch of P producer CTAs and C consumer CTAs, one CTA per SM, all
// co-resident:
//   producers  copy token rows into the gathered (or dispatched) buffer and
//              count them with the single-writer protocol of "cross-GPU sync
//              protocols on PCIe", sections 3-5 (producer.cuh);
//   consumers  run a tcgen05 bf16 GEMM over output tiles in row-block order,
//              gating the rows of each tile on the protocol with acquire
//              polls before loading them (consumer.cuh).
// Each chunk watermark may be split along K into k_slices sub-watermarks:
// the consumer's minimal release unit is a K-range of a row block, and the
// signal follows it (section 4: signal granularity follows the consumer's
// release unit).  Producers copy in the consumers' traversal order (section
// 6, item 3) so the first tiles start after a fraction of their rows has
// landed.  With k_slices = 1 each slot is exactly one 64-row chunk watermark.
// Producers never wait on anyone; consumers wait only on producers, which are
// resident by construction, and every wait is bounded.
//
// Instantiations: PAIR = 1 (one CTA per 128x256 tile) or 2 (a cluster pair
// per 256x256 tile with cta_group::2 MMAs), each with a fixed tile schedule
// or, DYN, the dynamic one of the role switch (tiles from a ticket counter,
// producers that turn consumer); and, EMB, a fixed schedule without producer
// CTAs whose consumer CTAs copy the rows in their spare warps.  Each variant
// is a kernel of its own so that the fixed-schedule kernel compiles without
// the others' roles.
#include <cuda_runtime.h>
#include "ctrl.cuh"
#include "ptx.cuh"
#include "sync.cuh"
#include "common.cuh"
#include "producer.cuh"
#include "consumer.cuh"
#include "launch.cuh"

namespace tovl {

template <int PAIR, bool DYN, bool EMB, int NW = 1>
__global__ void __launch_bounds__(kThreads, 1) fused_kernel(const __grid_constant__ FusedParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    if (static_cast<int>(blockIdx.x) < p.n_producers) {
        producer(p, smem, blockIdx.x);
        // role switch: with its copies done, the producer CTA (with its pair,
        // whose copies the consumer prologue's cluster barrier waits for)
        // takes GEMM tiles from the round's ticket counter like any consumer
        if (DYN && p.join) consumer<PAIR, DYN, false>(p, smem, -1);
    } else {
        consumer<PAIR, DYN, EMB, NW>(p, smem, blockIdx.x - p.n_producers);
    }
}

cudaError_t launch_fused(const FusedParams& p, cudaStream_t stream, bool cooperative, int pair, bool pdl)
{
    const int grid = p.n_producers + p.n_consumers;
    if (grid <= 0) return cudaSuccess;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(grid);
    lc.blockDim = dim3(kThreads);
    lc.dynamicSmemBytes = p.wide ? smem_bytes_wide() : p.embedded ? smem_bytes_emb(pair) : smem_bytes(pair);
    lc.stream = stream;
    cudaLaunchAttribute attr[3];
    int n = 0;
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n].val.cooperative = cooperative ? 1 : 0;
    ++n;
    if (pdl) {
        // the kernel's prologue may overlap the previous kernel's tail; every
        // role waits (griddepcontrol.wait) before it reads global memory
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (pair == 2) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = 2;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    lc.attrs = attr;
    lc.numAttrs = n;
    if (p.wide) return cudaLaunchKernelEx(&lc, fused_kernel<2, false, true, 2>, p);
    if (p.embedded)
        return pair == 2 ? cudaLaunchKernelEx(&lc, fused_kernel<2, false, true>, p)
                         : cudaLaunchKernelEx(&lc, fused_kernel<1, false, true>, p);
    if (pair == 2) return p.dyn ? cudaLaunchKernelEx(&lc, fused_kernel<2, true, false>, p)
                                : cudaLaunchKernelEx(&lc, fused_kernel<2, false, false>, p);
    return p.dyn ? cudaLaunchKernelEx(&lc, fused_kernel<1, true, false>, p)
                 : cudaLaunchKernelEx(&lc, fused_kernel<1, false, false>, p);
}

cudaError_t prepare_fused()
{
    cudaError_t e = cudaFuncSetAttribute(fused_kernel<1, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes(1));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fused_kernel<1, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes(1));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fused_kernel<2, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes(2));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fused_kernel<2, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes(2));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fused_kernel<1, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes_emb(1));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fused_kernel<2, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes_emb(2));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fused_kernel<2, false, true, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes_wide());
    return e;
}

int fused_max_active_per_sm()
{
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fused_kernel<1, false, false>, kThreads, smem_bytes(1)) != cudaSuccess)
        return 0;
    return n;
}

int fused_max_active_pairs()
{
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(2);
    lc.blockDim = dim3(kThreads);
    lc.dynamicSmemBytes = smem_bytes(2);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fused_kernel<2, false, false>, &lc) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace tovl
