// Backward kernels of the chunked gated delta rule (placeholder until written).
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace gdr {

cudaError_t launch_chain_bwd(const Args &, const void *, const void *, const float *, const void *, const void *,
                             const void *, const float *, void *, float *, cudaStream_t) {
    return cudaErrorNotSupported;
}
cudaError_t launch_bwd_chunk(const Args &, const void *, const void *, const void *, const float *, const void *,
                             const void *, const void *, const void *, const void *, void *, void *, void *, void *,
                             void *, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace gdr
