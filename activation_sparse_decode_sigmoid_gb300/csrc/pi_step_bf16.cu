// Instantiation of the step kernel for __nv_bfloat16 weights and activations
// (one translation unit per type, so that the three compile in parallel).
#include "pi_step.cuh"

namespace pi {

cudaError_t launch_step_bf16(const StepParams &p, int tgf, int grid, cudaStream_t s)
{
    return launch_step<__nv_bfloat16, false>(p, tgf, grid, s);
}

} // namespace pi
