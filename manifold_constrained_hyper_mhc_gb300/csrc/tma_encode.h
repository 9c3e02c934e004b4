// Host side of the TMA tensor copies: cuTensorMapEncodeTiled, fetched once from the driver
// through the runtime's entry-point query (no link against libcuda).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

namespace mhc {
namespace tma {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline cudaError_t encoder(EncodeTiledFn &fn) {
    static std::mutex mu;
    static EncodeTiledFn cached = nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (cached == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || p == nullptr) return cudaErrorNotSupported;
        cached = reinterpret_cast<EncodeTiledFn>(p);
    }
    fn = cached;
    return cudaSuccess;
}

// A bf16 tensor map with unit element strides and zero fill outside the tensor.
inline cudaError_t encode_bf16(EncodeTiledFn fn, CUtensorMap *m, int rank, const void *ptr, const cuuint64_t *dims,
                               const cuuint64_t *strides, const cuuint32_t *box, CUtensorMapSwizzle swz) {
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(ptr), dims, strides, box,
                    es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace tma
}  // namespace mhc
