// Recurrent decode of the gated delta rule: tokens applied one at a time to a cached fp32 state, the
// adjacent inference step of the chunked forward.  Per token (FlashQLA skill page, "Core API": the
// recurrence S_t = e^{g_t} S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T, o_t = scale S_t q_t), with
// h = S^T [K x V] and k, q optionally L2-normalised:
//
//   u  = h^T k                         (V-vector)
//   h <- e^{g} h + k (beta (v - e^{g} u))^T
//   o  = scale h^T q
//
// One CTA of 128 threads per (sequence, value head): thread v holds column v of h in 128 fp32 registers,
// so u and o are dot products inside a thread and every state row moves as one coalesced 512-byte access
// (the [V][K] layout: one contiguous 512-byte column per thread).  The kernel is bound by HBM: 64 KB of
// state read and 64 KB written per (sequence, head), plus 1 KB of token data per token.
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace gdr {
namespace {

constexpr int DN = 128;  // K = V = 128: one thread per value column, one key row per state element

struct DecArgs {
    const void *q, *k, *v, *g, *beta;
    const float *state_in;  // nullable: zero start
    float *state_out;       // may alias state_in
    void *o;
    int B, T, Hq, Hv;
    float scale;
    bool gate_f32, l2norm, v_first;
};

// Sum over the 128 threads of the block (fixed order: warp butterflies, then the four warp sums).
__device__ __forceinline__ float block_sum(float x, float *red, int lane, int warp) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0) red[warp] = x;
    __syncthreads();
    const float s = (red[0] + red[1]) + (red[2] + red[3]);
    __syncthreads();
    return s;
}

template <typename T>
__global__ void __launch_bounds__(DN) decode_kernel(const DecArgs a) {
    __shared__ __align__(16) float sq[DN];
    __shared__ __align__(16) float sk[DN];
    __shared__ float red[4];
    const int j = blockIdx.x, n = blockIdx.y, v = threadIdx.x;
    const int lane = v & 31, warp = v >> 5;
    const int hq = j / (a.Hv / a.Hq);
    const size_t sbase = ((size_t)n * a.Hv + j) * DN * DN;

    float h[DN];  // column v of h: h[d] = h_{d,v}
    if (a.state_in) {
        if (a.v_first) {
            const float4 *col = reinterpret_cast<const float4 *>(a.state_in + sbase + (size_t)v * DN);
#pragma unroll
            for (int i = 0; i < DN / 4; ++i) {
                const float4 x = col[i];
                h[4 * i] = x.x, h[4 * i + 1] = x.y, h[4 * i + 2] = x.z, h[4 * i + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int d = 0; d < DN; ++d) h[d] = a.state_in[sbase + (size_t)d * DN + v];
        }
    } else {
#pragma unroll
        for (int d = 0; d < DN; ++d) h[d] = 0.f;
    }

    const T *q = static_cast<const T *>(a.q);
    const T *k = static_cast<const T *>(a.k);
    const T *vv = static_cast<const T *>(a.v);
    T *o = static_cast<T *>(a.o);
    for (int t = 0; t < a.T; ++t) {
        const long long tk = ((long long)n * a.T + t) * a.Hq + hq;  // token row of q, k
        const long long tv = ((long long)n * a.T + t) * a.Hv + j;   // token row of v, g, beta, o
        const float qe = Elt<T>::to_f(q[tk * DN + v]), ke = Elt<T>::to_f(k[tk * DN + v]);
        const float ve = Elt<T>::to_f(vv[tv * DN + v]);
        const float gt = load_gate<T>(a.g, tv, a.gate_f32), bt = load_gate<T>(a.beta, tv, a.gate_f32);
        float rq = 1.f, rk = 1.f;
        if (a.l2norm) {
            rq = 1.0f / sqrtf(block_sum(qe * qe, red, lane, warp) + L2_EPS);
            rk = 1.0f / sqrtf(block_sum(ke * ke, red, lane, warp) + L2_EPS);
        }
        sq[v] = qe * rq;
        sk[v] = ke * rk;
        __syncthreads();
        const float4 *k4 = reinterpret_cast<const float4 *>(sk);
        const float4 *q4 = reinterpret_cast<const float4 *>(sq);
        float u = 0.f;
#pragma unroll
        for (int i = 0; i < DN / 4; ++i) {
            const float4 kk = k4[i];
            u = fmaf(h[4 * i], kk.x, u);
            u = fmaf(h[4 * i + 1], kk.y, u);
            u = fmaf(h[4 * i + 2], kk.z, u);
            u = fmaf(h[4 * i + 3], kk.w, u);
        }
        const float e = __expf(gt);
        const float w = bt * (ve - e * u);
        float ov = 0.f;
#pragma unroll
        for (int i = 0; i < DN / 4; ++i) {
            const float4 kk = k4[i], qq = q4[i];
            h[4 * i] = fmaf(e, h[4 * i], kk.x * w);
            h[4 * i + 1] = fmaf(e, h[4 * i + 1], kk.y * w);
            h[4 * i + 2] = fmaf(e, h[4 * i + 2], kk.z * w);
            h[4 * i + 3] = fmaf(e, h[4 * i + 3], kk.w * w);
            ov = fmaf(h[4 * i], qq.x, ov);
            ov = fmaf(h[4 * i + 1], qq.y, ov);
            ov = fmaf(h[4 * i + 2], qq.z, ov);
            ov = fmaf(h[4 * i + 3], qq.w, ov);
        }
        o[tv * DN + v] = Elt<T>::from_f(a.scale * ov);
        __syncthreads();  // sq, sk are rewritten by the next token
    }

    if (a.v_first) {
        float4 *col = reinterpret_cast<float4 *>(a.state_out + sbase + (size_t)v * DN);
#pragma unroll
        for (int i = 0; i < DN / 4; ++i) col[i] = make_float4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
    } else {
#pragma unroll
        for (int d = 0; d < DN; ++d) a.state_out[sbase + (size_t)d * DN + v] = h[d];
    }
}

template <typename T>
cudaError_t decode_t(const DecArgs &d, cudaStream_t s) {
    decode_kernel<T><<<dim3(d.Hv, d.B), DN, 0, s>>>(d);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const Args &a, const void *q, const void *k, const void *v, const void *g,
                          const void *beta, const float *state_in, float *state_out, void *o, cudaStream_t s) {
    DecArgs d;
    d.q = q;
    d.k = k;
    d.v = v;
    d.g = g;
    d.beta = beta;
    d.state_in = state_in;
    d.state_out = state_out;
    d.o = o;
    d.B = a.B;
    d.T = a.T;
    d.Hq = a.Hq;
    d.Hv = a.Hv;
    d.scale = a.scale;
    d.gate_f32 = a.gate_f32;
    d.l2norm = a.l2norm;
    d.v_first = a.v_first;
    return a.bf16 ? decode_t<__nv_bfloat16>(d, s) : decode_t<__half>(d, s);
}

}  // namespace gdr
