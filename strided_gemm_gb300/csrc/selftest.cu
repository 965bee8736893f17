// Self-test of the failure detection every kernel path relies on: a bounded
// wait that runs out records a code in a device status word and the kernel
// returns, so the context stays usable and sbgemm_device_status reports
// SBGEMM_ERR_DEVICE_TIMEOUT.  The waits here are the same helpers the kernels
// use (mbar_wait, wait_flag), given a short limit, on conditions that nothing
// will ever satisfy.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "sbgemm.h"

namespace sbg {
namespace {

__device__ unsigned int g_wait_status = 0;
__device__ unsigned int g_never_set = 0;    // a flag no code writes

__global__ void selftest_kernel(int what, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (what == SBGEMM_SELFTEST_MBARRIER) {
        // Phase 0 needs one arrival that no thread makes.
        if (!mbar_wait(&bar, 0, limit_ns)) record_status(&g_wait_status, kWaitSelftestMbar);
    } else if (what == SBGEMM_SELFTEST_FLAG) {
        if (threadIdx.x == 0 && !wait_flag(&g_never_set, limit_ns))
            record_status(&g_wait_status, kWaitSelftestFlag);
    }
}

}  // namespace

unsigned int read_and_clear_wait_status_selftest(cudaStream_t stream) {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_wait_status, sizeof(v), 0, cudaMemcpyDeviceToHost,
                                  stream) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_wait_status, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice,
                                stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return v;
}

}  // namespace sbg

extern "C" int sbgemm_selftest(int what, int64_t limit_us, void* stream) {
    if (what != SBGEMM_SELFTEST_MBARRIER && what != SBGEMM_SELFTEST_FLAG) return SBGEMM_ERR_INVALID_VALUE;
    if (limit_us < 1 || limit_us > 2000000) return SBGEMM_ERR_INVALID_VALUE;
    sbg::selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        what, (uint64_t)limit_us * 1000u);
    if (cudaGetLastError() != cudaSuccess) return SBGEMM_ERR_CUDA;
    return SBGEMM_OK;
}
