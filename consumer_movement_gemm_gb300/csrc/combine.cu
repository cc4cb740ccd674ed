// combine.cu -- the combine kernel: producer CTAs stage expert-output rows in
// token order with per-chunk watermarks, reducer CTAs wait on the watermarks
// and write the gate-weighted sums.  One persistent grid, every CTA resident
// (cooperative launch), so a reducer's wait always has a live producer.
#include "combine.cuh"
#include "launch.cuh"
#include "producer.cuh"

namespace tovl {

__global__ void __launch_bounds__(kThreads, 1) combine_kernel(const __grid_constant__ FusedParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    // the expert outputs and the plan come from the kernels before this one
    ptx::grid_dep_wait();
    if (p.embedded > 0) {
        // every CTA copies in its first p.embedded warps and reduces in the
        // rest; copy items and tokens are dealt across all CTAs
        const int warp = threadIdx.x / 32;
        const int grid = static_cast<int>(gridDim.x);
        if (warp < p.embedded) {
            const int gw = warp * grid + static_cast<int>(blockIdx.x);
            const int n_gw = p.embedded * grid;
            seed_counters(p, gw, n_gw, true);
            if (p.item_rows <= 16) copy_items<1>(p, gw, n_gw);
            else if (p.item_rows == 32) copy_items<2>(p, gw, n_gw);
            else copy_items<4>(p, gw, n_gw);
            seed_counters(p, gw, n_gw, false);
        } else {
            reducer(p, static_cast<int>(blockIdx.x), grid, p.embedded);
        }
        return;
    }
    if (static_cast<int>(blockIdx.x) < p.n_producers) producer(p, smem, blockIdx.x);
    else reducer(p, blockIdx.x - p.n_producers, p.n_reducers, 0);
}

// Shared memory: the staged producer path keeps one 8 KB buffer and one
// mbarrier per warp; the vector path needs none, which leaves the SM's whole
// L1 to the copies.
static int combine_smem(int producer_mode)
{
    return producer_mode == 1 ? (kThreads / 32) * (kItemBytes + 8) + 1024 : 0;
}

cudaError_t prepare_combine()
{
    return cudaFuncSetAttribute(combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, combine_smem(1));
}

cudaError_t launch_combine(const FusedParams& p, cudaStream_t stream, bool cooperative, bool pdl)
{
    const int grid = p.n_producers + p.n_reducers;
    if (grid <= 0) return cudaSuccess;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(grid);
    lc.blockDim = dim3(kThreads);
    lc.dynamicSmemBytes = combine_smem(p.producer_mode);
    lc.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = cooperative ? 1 : 0;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&lc, combine_kernel, p);
}

}  // namespace tovl
