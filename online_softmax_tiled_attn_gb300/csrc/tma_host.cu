// tma_host.cu -- host-side TMA tensor-map encoding.
//
// cuTensorMapEncodeTiled is a CUDA driver function; it is fetched once through the runtime's
// versioned entry-point query so the library does not link libcuda directly (it still loads
// on a machine without a GPU driver, and fails with FA_ERR_CUDA only when called).
#include <cudaTypedefs.h>

#include <mutex>

#include "osm_internal.h"

namespace osm {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

}  // namespace

int make_bhnd_tensor_map(CUtensorMap* map, const void* base, int64_t BH, int64_t N, int64_t d) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return FA_ERR_CUDA;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                   static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                     strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

int make_mask_tensor_map(CUtensorMap* map, const uint32_t* mask, int64_t W, int64_t Nq,
                         int64_t Hm, int64_t Bm, int64_t mask_hs, int64_t mask_bs) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return FA_ERR_CUDA;
    // A dimension of one instance takes the dense stride (it is only ever indexed at 0).
    const cuuint64_t row = static_cast<cuuint64_t>(W) * 4;
    const cuuint64_t hs = Hm > 1 ? static_cast<cuuint64_t>(mask_hs) * 4 : row * Nq;
    const cuuint64_t bs = Bm > 1 ? static_cast<cuuint64_t>(mask_bs) * 4 : hs * Hm;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(W), static_cast<cuuint64_t>(Nq),
                                static_cast<cuuint64_t>(Hm), static_cast<cuuint64_t>(Bm)};
    const cuuint64_t strides[3] = {row, hs, bs};
    const cuuint32_t box[4] = {4, 128, 1, 1};  // one key tile's 128 bits for 128 query rows
    const cuuint32_t estride[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, const_cast<uint32_t*>(mask), dims,
                     strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

}  // namespace osm
