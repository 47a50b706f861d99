// Host side of the TMA tensor maps the kernels copy their tiles with.
//
// The driver's cuTensorMapEncodeTiled is reached through the runtime's
// driver entry-point query once per process (no link against libcuda).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.h"

namespace lora {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

cudaError_t get_encoder() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                        cudaEnableDefault, &q);
        if (g_encode_err == cudaSuccess && (q != cudaDriverEntryPointSuccess || fn == nullptr))
            g_encode_err = cudaErrorNotSupported;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode_err;
}

}  // namespace

cudaError_t make_tensor_map_2d(CUtensorMap *m, lora_dtype_t dt, const void *base, uint64_t rows,
                               uint64_t cols, uint64_t ld, uint32_t box_rows) {
    cudaError_t e = get_encoder();
    if (e != cudaSuccess) return e;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {64u, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, dt == LORA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                          2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace lora
