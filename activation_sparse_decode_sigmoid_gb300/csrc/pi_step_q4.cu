// Instantiation of the step kernel for __half activations with Q4_0 FFN weights
// (one translation unit per type, so that the three compile in parallel).
#include "pi_step.cuh"

namespace pi {

cudaError_t launch_step_q4(const StepParams &p, int tgf, int grid, cudaStream_t s)
{
    return launch_step<__half, true>(p, tgf, grid, s);
}

} // namespace pi
