// Instantiation of the step kernel for __half weights and activations
// (one translation unit per type, so that the three compile in parallel).
#include "pi_step.cuh"

namespace pi {

cudaError_t launch_step_f16(const StepParams &p, int tgf, int grid, cudaStream_t s)
{
    return launch_step<__half, false>(p, tgf, grid, s);
}

} // namespace pi
