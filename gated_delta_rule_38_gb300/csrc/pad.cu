// Head dimensions below 128: the chunked kernels are written for K = V = 128 and run smaller problems as if
// zero-padded.  Padding is exact for this recurrence: zero key coordinates leave k.k, q.k and the L2 norms
// unchanged and keep the state's padded rows zero; zero value coordinates keep its padded columns zero; so
// the padded outputs hold the true ones in their leading K / V coordinates and zeros elsewhere.  The token
// tensors need no copies (the kernels' TMA boxes load zeros past K / V); these kernels copy the fp32 state
// tensors [NH, R, Cc] <-> [NH, 128, 128] (Cc a multiple of 4), zero-filling on the way in.
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace gdr {
namespace {

inline unsigned grid_for(long long n) {
    const long long b = (n + 255) / 256;
    return (unsigned)(b < 8192 ? (b > 0 ? b : 1) : 8192);
}

// fp32 states: one thread per float4 of the padded [128][128] matrix.
__global__ void pad_state_kernel(const float4 *__restrict__ src, float4 *__restrict__ dst, long long nh, int R,
                                 int c4) {
    griddep_wait();
    const long long n = nh * 128 * 32;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const long long m = i / (128 * 32);
        const int rem = (int)(i - m * 128 * 32), r = rem >> 5, c = rem & 31;
        dst[i] = (r < R && c < c4) ? src[(m * R + r) * c4 + c] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

__global__ void unpad_state_kernel(const float4 *__restrict__ src, float4 *__restrict__ dst, long long nh, int R,
                                   int c4) {
    griddep_wait();
    const long long n = nh * R * c4;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const long long m = i / ((long long)R * c4);
        const int rem = (int)(i - m * R * c4), r = rem / c4, c = rem - r * c4;
        dst[i] = src[(m * 128 + r) * 32 + c];
    }
}

}  // namespace

cudaError_t launch_pad_state(const float *src, float *dst, long long nh, int R, int Cc, cudaStream_t s) {
    if (nh == 0) return cudaSuccess;
    return launch_plain(pad_state_kernel, dim3(grid_for(nh * 128 * 32)), dim3(256), 0, s,
                        reinterpret_cast<const float4 *>(src), reinterpret_cast<float4 *>(dst), nh, R, Cc / 4);
}

cudaError_t launch_unpad_state(const float *src, float *dst, long long nh, int R, int Cc, cudaStream_t s) {
    if (nh == 0) return cudaSuccess;
    return launch_plain(unpad_state_kernel, dim3(grid_for(nh * R * (Cc / 4))), dim3(256), 0, s,
                        reinterpret_cast<const float4 *>(src), reinterpret_cast<float4 *>(dst), nh, R, Cc / 4);
}

}  // namespace gdr
