// Driver API entry points fetched through the runtime, so the library needs no
// link-time dependency on libcuda.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace sbg {
namespace {

using MemGetAddressRangeFn = CUresult (*)(CUdeviceptr*, size_t*, CUdeviceptr);
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

MemGetAddressRangeFn g_mem_range = nullptr;
EncodeTiledFn g_encode_tiled = nullptr;
std::once_flag g_once;

void* entry_point(const char* name) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion(name, &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return fn;
    cudaGetLastError();
    return nullptr;
}

void load_entry_points() {
    g_mem_range = reinterpret_cast<MemGetAddressRangeFn>(entry_point("cuMemGetAddressRange"));
    g_encode_tiled = reinterpret_cast<EncodeTiledFn>(entry_point("cuTensorMapEncodeTiled"));
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

bool encode_tmap_f32_3d(CUtensorMap* map, const void* base, const uint64_t dims[3],
                        const uint64_t strides_bytes[2], const uint32_t box[3], bool swizzle128) {
    std::call_once(g_once, load_entry_points);
    if (!g_encode_tiled) return false;
    const cuuint64_t gdim[3] = {dims[0], dims[1], dims[2]};
    const cuuint64_t gstride[2] = {strides_bytes[0], strides_bytes[1]};
    const cuuint32_t bdim[3] = {box[0], box[1], box[2]};
    const cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base),
                                gdim, gstride, bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace sbg
