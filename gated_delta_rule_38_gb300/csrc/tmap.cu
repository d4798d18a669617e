// TMA tensor maps for the kernels' tile loads.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "tmap.h"

namespace gdr {
namespace {

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

using CtxGetFn = CUresult (*)(CUcontext *);

void *driver_symbol(const char *name) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return p;
    return nullptr;
}

EncodeFn encoder() {
    static std::once_flag once;
    static EncodeFn fn = nullptr;
    std::call_once(once, [] { fn = reinterpret_cast<EncodeFn>(driver_symbol("cuTensorMapEncodeTiled")); });
    return fn;
}

CtxGetFn ctx_get() {
    static std::once_flag once;
    static CtxGetFn fn = nullptr;
    std::call_once(once, [] { fn = reinterpret_cast<CtxGetFn>(driver_symbol("cuCtxGetCurrent")); });
    return fn;
}

}  // namespace

cudaError_t ensure_context() {
    CtxGetFn get = ctx_get();
    if (!get) return cudaErrorInitializationError;
    CUcontext c = nullptr;
    if (get(&c) != CUDA_SUCCESS) return cudaErrorInitializationError;
    if (c) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    return cudaSetDevice(dev);
}

bool make_tmap_3d(CUtensorMap *map, const void *base, bool bf16, uint64_t dim0, uint64_t dim1, uint64_t dim2,
                  uint64_t stride1, uint64_t stride2, uint32_t box0, uint32_t box1, uint32_t box2) {
    EncodeFn enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {dim0, dim1, dim2 > 0 ? dim2 : 1};
    const cuuint64_t strides[2] = {stride1, stride2};
    const cuuint32_t box[3] = {box0, box1, box2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base),
               dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace gdr
