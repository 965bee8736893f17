// sbgemm_noalloc: the product for callers that cannot allocate device memory.
//
// The stream-K schedule of the TMA FFMA kernel needs scratch (partial sums
// of split tiles and their ready flags), and so do the gather kernel's K
// pieces of small products.  sbgemm_ex takes that scratch from the caller.
// Some callers have no way to provide it:
//  - code that runs while a CUDA graph is being captured, where cudaMalloc
//    is not allowed;
//  - a plugin that the host application hands only its input and output
//    buffers;
//  - a latency-critical loop that must not pay cudaMalloc's implicit
//    synchronisation;
//  - a runtime whose allocator owns all device memory.
// This entry point gives them the same kernels with scratch that belongs to
// the library: a file-scope array in device memory, created once when the
// module is loaded and held by every GPU that loads the library until the
// process exits.
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
constexpr size_t kNoAllocScratchBytes = SBGEMM_NOALLOC_SCRATCH_BYTES;

static_assert(kNoAllocScratchBytes >= (size_t)kNoAllocMaxSms * kWorkspaceBytesPerSm,
              "the schedule's scratch for a device of kNoAllocMaxSms SMs");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_lookup_mutex;
std::array<void*, kMaxDevices> g_scratch{};   // written under the mutex, once non-null never again

// Device address of the scratch array on the current device, or nullptr if
// it could not be looked up.  In host code the array's name is only a
// host-side handle, so the address is looked up with the device current.
// Only a successful lookup is kept: a failed one (say, a transient error) is
// retried by the next call.  A lookup may load the library's module on the
// device, which a stream being captured must not see, so the first call on a
// device is refused while `stream` is capturing.
int scratch_address(int dev, cudaStream_t stream, void** out) {
    std::lock_guard<std::mutex> lock(g_lookup_mutex);
    if (g_scratch[dev]) {
        *out = g_scratch[dev];
        return SBGEMM_OK;
    }
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
        cudaGetLastError();
        return SBGEMM_ERR_CUDA;
    }
    if (cap != cudaStreamCaptureStatusNone) return SBGEMM_ERR_CUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return SBGEMM_ERR_CUDA;
    }
    g_scratch[dev] = p;
    *out = p;
    return SBGEMM_OK;
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
    void* scratch = nullptr;
    st = sbg::scratch_address(dev, static_cast<cudaStream_t>(stream), &scratch);
    if (st != SBGEMM_OK) return st;
    sbgemm_options o{};
    o.math = SBGEMM_MATH_FP32;
    o.force_path = SBGEMM_PATH_AUTO;
    o.k_split = SBGEMM_KSPLIT_ANY;
    o.workspace = scratch;
    o.workspace_bytes = sbg::kNoAllocScratchBytes;
    return sbgemm_ex(A, rsA, csA, bsA, B, rsB, csB, bsB, C, rsC, csC, bsC,
                     M, N, K, batch, alpha, accumulate, stream, &o);
}
