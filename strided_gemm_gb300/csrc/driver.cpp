// Driver API entry points fetched through the runtime, so the library needs no
// link-time dependency on libcuda.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace sbg {
namespace {

using MemGetAddressRangeFn = CUresult (*)(CUdeviceptr*, size_t*, CUdeviceptr);

MemGetAddressRangeFn g_mem_range = nullptr;
std::once_flag g_once;

void load_entry_points() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
        g_mem_range = reinterpret_cast<MemGetAddressRangeFn>(fn);
    }
}

}  // namespace

bool device_allocation_range(const void* ptr, uintptr_t* base, size_t* size) {
    std::call_once(g_once, load_entry_points);
    if (!g_mem_range) return false;
    CUdeviceptr b = 0;
    size_t s = 0;
    if (g_mem_range(&b, &s, reinterpret_cast<CUdeviceptr>(ptr)) != CUDA_SUCCESS) return false;
    *base = static_cast<uintptr_t>(b);
    *size = s;
    return true;
}

}  // namespace sbg
