// The TMA-fed FFMA kernels with 128 x 256 tiles (ffma_tma_kernel.cuh), one
// translation unit per tile shape.
#include "ffma_tma_kernel.cuh"

namespace sbg {

cudaError_t launch_tma_ffma_128x256(const Problem& p, const Plan& plan, int sm_count,
                                   cudaStream_t stream) {
    return launch_tile<128, 256>(p, plan, sm_count, stream);
}

unsigned int read_and_clear_wait_status_tma_ffma_128x256(cudaStream_t stream) {
    return read_and_clear_status(stream);
}

}  // namespace sbg
