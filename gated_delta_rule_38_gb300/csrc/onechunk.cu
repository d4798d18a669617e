// The dg of sequences that fit in one chunk, with an initial state and a final-state gradient.
//
// The per-chunk gradient kernel adds e^{G_last} <dH', h> (the decay term of the state that the chunk carries
// over) at the chunk's last valid row, and its reverse cumsum passes it to every row.  It takes h and dH' from
// their tiles in the input dtype.  For a sequence of one chunk those are the caller's h0 and dht, and that term
// is most of the sequence's dg (the other terms are over one chunk only), so the tiles' rounding shows there
// (one token, K = V = 128: 2 % relative in dg).  This kernel adds to such a sequence's dg, at every row, the
// difference e^{G_last} (<dht, h0> - <rounded dht, rounded h0>) computed in fp32 from the caller's states.
// One block of 1024 threads per (sequence, value head); a block whose sequence has no chunk or more than one
// returns at once.
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace gdr {
namespace {

template <typename T>
__device__ __forceinline__ float rounded(float x) {
    return Elt<T>::to_f(Elt<T>::from_f(x));
}

template <typename T>
__global__ void __launch_bounds__(1024) onechunk_dg_kernel(Geo geo, const float *__restrict__ h0,
                                                          const float *__restrict__ dht, const float *__restrict__ g_cs,
                                                          void *dg, bool dg_f32) {
    griddep_wait();
    __shared__ float red[2][32];
    const int Hv = geo.Hv, j = (int)(blockIdx.x % (unsigned)Hv), n = (int)(blockIdx.x / (unsigned)Hv);
    long long tok0;
    int len, row0;
    geo.seq(n, tok0, len, row0);
    if (len <= 0 || len > C) return;
    const long long base = ((long long)n * Hv + j) * DK * DV;
    const float4 *a4 = reinterpret_cast<const float4 *>(h0 + base);
    const float4 *b4 = reinterpret_cast<const float4 *>(dht + base);
    float exact = 0.f, tile = 0.f;
#pragma unroll
    for (int u = 0; u < DK * DV / 4 / 1024; ++u) {  // (every load in flight at once)
        const int i = u * 1024 + (int)threadIdx.x;
        const float4 a = a4[i], b = b4[i];
        exact += a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
        tile += rounded<T>(a.x) * rounded<T>(b.x) + rounded<T>(a.y) * rounded<T>(b.y) +
                rounded<T>(a.z) * rounded<T>(b.z) + rounded<T>(a.w) * rounded<T>(b.w);
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        exact += __shfl_xor_sync(0xffffffffu, exact, o);
        tile += __shfl_xor_sync(0xffffffffu, tile, o);
    }
    if (lane == 0) {
        red[0][warp] = exact;
        red[1][warp] = tile;
    }
    __syncthreads();
    if ((int)threadIdx.x >= len) return;
    float e = 0.f, t = 0.f;
#pragma unroll
    for (int w = 0; w < 32; ++w) {
        e += red[0][w];
        t += red[1][w];
    }
    const float delta = __expf(g_cs[(tok0 + len - 1) * Hv + j]) * (e - t);
    const long long ti = (tok0 + threadIdx.x) * Hv + j;
    store_gate<T>(dg, ti, dg_f32, load_gate<T>(dg, ti, dg_f32) + delta);
}

}  // namespace

cudaError_t launch_onechunk_dg(const Args &a, const float *h0, const float *dht, const float *g_cs, void *dg,
                               cudaStream_t s) {
    const long long blocks = (long long)a.N * a.Hv;
    if (blocks == 0) return cudaSuccess;
    // (may begin launching while the per-chunk gradients finish: it waits for them before touching memory)
    if (a.bf16)
        return launch_overlapped(onechunk_dg_kernel<__nv_bfloat16>, dim3((unsigned)blocks), dim3(1024), 0, s,
                                 make_geo(a), h0, dht, g_cs, dg, a.gate_f32);
    return launch_overlapped(onechunk_dg_kernel<__half>, dim3((unsigned)blocks), dim3(1024), 0, s, make_geo(a), h0,
                             dht, g_cs, dg, a.gate_f32);
}

}  // namespace gdr
