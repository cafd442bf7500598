// Host side of the tensor-core kernels: the tensor-map encoder, looked up once through the
// runtime's driver entry point (no link against the driver library).
#include <cudaTypedefs.h>

#include <mutex>

#include "prox_tc.cuh"

namespace prox {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

int encode_map_2d(CUtensorMap* tm, CUtensorMapDataType type, const void* base, uint64_t cols,
                  uint64_t rows, uint64_t pitch, uint32_t box_cols, uint32_t box_rows,
                  CUtensorMapSwizzle swizzle) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cuda_fail(cudaErrorNotSupported, "looking up cuTensorMapEncodeTiled");
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {pitch};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(tm, type, 2, const_cast<void*>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PROX_OK : cuda_fail(cudaErrorInvalidValue, "encoding a tensor map");
}

}  // namespace prox
