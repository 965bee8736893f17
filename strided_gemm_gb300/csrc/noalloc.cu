// sbgemm_noalloc: the product for callers that cannot allocate device memory.
//
// The stream-K schedule of the TMA FFMA kernel needs scratch (partial sums
// of split tiles and their ready flags).  sbgemm_ex takes that scratch from
// the caller.  Some callers have no way to provide it:
//  - code that runs while a CUDA graph is being captured, where cudaMalloc
//    is not allowed;
//  - a plugin that the host application hands only its input and output
//    buffers;
//  - a latency-critical loop that must not pay cudaMalloc's implicit
//    synchronisation;
//  - a runtime whose allocator owns all device memory.
// This entry point gives them the same kernel with scratch that belongs to the
// library: a file-scope array in device memory, created once when the module
// is loaded and held by every GPU that loads the library until the process
// exits.
#include <cuda_runtime.h>

#include <array>
#include <mutex>

#include "internal.h"
#include "sbgemm.h"

namespace sbg {
namespace {

// Capacity: the stream-K scratch of a device with up to 160 SMs (one fp32
// partial tile per SM plus one flag word per SM); 20 MiB + 4 KiB.
constexpr int kNoAllocMaxSms = 160;
constexpr size_t kNoAllocScratchBytes = (size_t)20 * 1024 * 1024 + 4096;

static_assert(kNoAllocScratchBytes >= (size_t)kNoAllocMaxSms * (256 * 64 * 8 + 4),
              "one partial tile (256 threads x 64 float pairs) and one flag per SM");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::array<std::once_flag, kMaxDevices> g_once;
std::array<void*, kMaxDevices> g_scratch{};
std::array<cudaError_t, kMaxDevices> g_scratch_err{};

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side handle, so the address is looked up
// once per device, with that device current.
void* scratch_address(int dev) {
    std::call_once(g_once[dev], [dev] {
        void* p = nullptr;
        g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        g_scratch[dev] = p;
        if (g_scratch_err[dev] != cudaSuccess) cudaGetLastError();
    });
    return g_scratch_err[dev] == cudaSuccess ? g_scratch[dev] : nullptr;
}

}  // namespace
}  // namespace sbg

extern "C" int sbgemm_noalloc(const float* A, int64_t rsA, int64_t csA, int64_t bsA,
                              const float* B, int64_t rsB, int64_t csB, int64_t bsB,
                              float* C, int64_t rsC, int64_t csC, int64_t bsC,
                              int64_t M, int64_t N, int64_t K, int64_t batch,
                              float alpha, int accumulate, void* stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SBGEMM_ERR_CUDA;
    }
    if (dev < 0 || dev >= sbg::kMaxDevices) return SBGEMM_ERR_CUDA;
    size_t need = 0;
    int st = sbgemm_workspace_bytes(dev, &need);
    if (st != SBGEMM_OK) return st;
    // A device with more SMs than the array was sized for would need more
    // scratch than it holds.
    if (need > sbg::kNoAllocScratchBytes) return SBGEMM_ERR_UNSUPPORTED;
    void* scratch = sbg::scratch_address(dev);
    if (!scratch) return SBGEMM_ERR_CUDA;
    sbgemm_options o{};
    o.math = SBGEMM_MATH_FP32;
    o.force_path = SBGEMM_PATH_AUTO;
    o.workspace = scratch;
    o.workspace_bytes = sbg::kNoAllocScratchBytes;
    return sbgemm_ex(A, rsA, csA, bsA, B, rsB, csB, bsB, C, rsC, csC, bsC,
                     M, N, K, batch, alpha, accumulate, stream, &o);
}
