// Host-side construction of TMA tensor maps.  The driver entry point is
// looked up through the runtime once, so the library does not link libcuda.
#include <cudaTypedefs.h>

#include <mutex>

#include "opam_internal.cuh"
#include "sm100.cuh"

namespace opam {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

bool have_encode() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                        cudaEnableDefault, &q);
        if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode) set_error("cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(g_encode_err));
    return g_encode != nullptr;
}

}  // namespace

int make_tmap_bf16_3d(CUtensorMap *map, const void *base, uint64_t n0, uint64_t n1, uint64_t n2,
                      uint32_t box1) {
    if (!have_encode()) return OPAM_ERR_CUDA;
    const cuuint64_t dims[3] = {n0, n1, n2};
    const cuuint64_t strides[2] = {n0 * 2, n0 * n1 * 2};  // bytes, dims 1 and 2
    const cuuint32_t box[3] = {64, box1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (%d) for dims {%llu, %llu, %llu} box {64, %u, 1}",
                  (int)r, (unsigned long long)n0, (unsigned long long)n1, (unsigned long long)n2,
                  box1);
        return OPAM_ERR_INVALID_ARG;
    }
    return OPAM_OK;
}

int make_tmap_f32_3d(CUtensorMap *map, const void *base, uint64_t n0, uint64_t n1, uint64_t n2,
                     uint32_t box0, uint32_t box1) {
    if (!have_encode()) return OPAM_ERR_CUDA;
    const cuuint64_t dims[3] = {n0, n1, n2};
    const cuuint64_t strides[2] = {n0 * 4, n0 * n1 * 4};  // bytes, dims 1 and 2
    const cuuint32_t box[3] = {box0, box1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (%d) for float32 dims {%llu, %llu, %llu} box {%u, %u, 1}", (int)r,
                  (unsigned long long)n0, (unsigned long long)n1, (unsigned long long)n2, box0, box1);
        return OPAM_ERR_INVALID_ARG;
    }
    return OPAM_OK;
}

}  // namespace opam
