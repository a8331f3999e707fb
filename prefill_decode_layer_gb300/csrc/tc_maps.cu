// Host side of the tensor-core GEMM: TMA tensor maps (cuTensorMapEncodeTiled, from
// the driver through the runtime's entry-point query; no link to libcuda).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "tc_gemm.cuh"

namespace ds4g {
namespace tc {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

cudaError_t make_map_bf16(CUtensorMap *m, const void *base, int rows, int cols, int ld, int box_rows)
{
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    if (rows <= 0 || cols <= 0 || ld < cols || ((uintptr_t)base & 15u) || (ld * 2) % 16 || box_rows > 256)
        return cudaErrorInvalidValue;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace tc
}  // namespace ds4g
