// tmap.cu -- host-side TMA tensor-map encoding (cuTensorMapEncodeTiled through
// the runtime's driver entry point, so the library does not link libcuda).
#include <cudaTypedefs.h>

#include <mutex>

#include "tmap.cuh"

namespace ssd {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;

void init_encode() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    else
        cudaGetLastError();
}

}  // namespace

bool make_tmap_16b_4d(CUtensorMap* map, const void* base, const uint64_t dims[4], const uint32_t box[4]) {
    std::call_once(g_once, init_encode);
    if (g_encode == nullptr) return false;
    cuuint64_t gdim[4] = {dims[0], dims[1], dims[2], dims[3]};
    cuuint64_t gstride[3] = {dims[0] * 2, dims[0] * dims[1] * 2, dims[0] * dims[1] * dims[2] * 2};
    cuuint32_t bdim[4] = {box[0], box[1], box[2], box[3]};
    cuuint32_t estride[4] = {1, 1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void*>(base), gdim, gstride, bdim,
                          estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace ssd
