// The TMA-fed FFMA kernels with 512 x 64 tiles (ffma_tma_kernel.cuh), one
// translation unit per tile shape.
#include "ffma_tma_kernel.cuh"

namespace sbg {

cudaError_t launch_tma_ffma_512x64(const Problem& p, const Plan& plan, int sm_count,
                                   cudaStream_t stream) {
    // Planned only for a K-major A (tma_ffma_pick_variant): the 512-row A of
    // an MN-major operand would not fit one TMA box.
    if (plan.a_layout != SBGEMM_LAYOUT_K_MAJOR) return cudaErrorInvalidValue;
    if (plan.b_layout == SBGEMM_LAYOUT_K_MAJOR)
        return launch_impl<512, 64, true, true>(p, plan, sm_count, stream);
    return launch_impl<512, 64, true, false>(p, plan, sm_count, stream);
}

unsigned int read_and_clear_wait_status_tma_ffma_512x64(cudaStream_t stream) {
    return read_and_clear_status(stream);
}

}  // namespace sbg
