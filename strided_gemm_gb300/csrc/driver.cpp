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

namespace {

bool encode_tmap_f32(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides_bytes, const uint32_t* box, bool swizzle128) {
    std::call_once(g_once, load_entry_points);
    if (!g_encode_tiled || rank < 1 || rank > 5) return false;
    cuuint64_t gdim[5], gstride[4];
    cuuint32_t bdim[5], estride[5];
    for (int i = 0; i < rank; ++i) {
        gdim[i] = dims[i];
        bdim[i] = box[i];
        estride[i] = 1;
        if (i + 1 < rank) gstride[i] = strides_bytes[i];
    }
    CUresult r = g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (cuuint32_t)rank, const_cast<void*>(base),
                                gdim, gstride, bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

bool encode_tmap_f32_3d(CUtensorMap* map, const void* base, const uint64_t dims[3],
                        const uint64_t strides_bytes[2], const uint32_t box[3], bool swizzle128) {
    return encode_tmap_f32(map, base, 3, dims, strides_bytes, box, swizzle128);
}

bool encode_tmap_f32_4d(CUtensorMap* map, const void* base, const uint64_t dims[4],
                        const uint64_t strides_bytes[3], const uint32_t box[4], bool swizzle128) {
    return encode_tmap_f32(map, base, 4, dims, strides_bytes, box, swizzle128);
}

}  // namespace sbg
