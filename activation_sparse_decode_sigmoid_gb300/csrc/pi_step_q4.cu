// Instantiation of the step kernel for __half activations with Q4_0 FFN weights.
#include "pi_step.cuh"

namespace pi {

template <int TGF> static cudaError_t launch_tgf(const StepParams &p, int grid, cudaStream_t s)
{
    auto kern = step_kernel<__half, true, TGF>;
    static int configured = -1; // dynamic shared memory the attribute was last set to
    if (configured != p.smem_bytes) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes);
        if (e != cudaSuccess) return e;
        configured = p.smem_bytes;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = p.smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_step_q4(const StepParams &p, int tgf, int grid, cudaStream_t s)
{
    return tgf == 1 ? launch_tgf<1>(p, grid, s) : tgf == 2 ? launch_tgf<2>(p, grid, s) : launch_tgf<4>(p, grid, s);
}

cudaError_t occupancy_step_q4(int tgf, int smem_bytes, int *blocks)
{
    if (tgf == 1)
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, step_kernel<__half, true, 1>, kThreads, smem_bytes);
    if (tgf == 2)
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, step_kernel<__half, true, 2>, kThreads, smem_bytes);
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, step_kernel<__half, true, 4>, kThreads, smem_bytes);
}

} // namespace pi
