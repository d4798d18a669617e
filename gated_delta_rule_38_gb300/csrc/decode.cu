// Recurrent decode of the gated delta rule: tokens applied one at a time to a cached fp32 state, the
// adjacent inference step of the chunked forward.  Per token (FlashQLA skill page, "Core API": the
// recurrence S_t = e^{g_t} S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T, o_t = scale S_t q_t), with
// h = S^T [K x V] and k, q optionally L2-normalised:
//
// (g and beta after the optional activations of GDR_GATE_IN_KERNEL / GDR_BETA_SIGMOID_IN_KERNEL /
// GDR_ALLOW_NEG_EIGVAL)
//   u  = h^T k                         (V-vector)
//   h <- e^{g} h + k (beta (v - e^{g} u))^T
//   o  = scale h^T q
//
// Head dims K, V <= 128: threads of columns v >= V and state rows d >= K hold zeros (exact: zero key
// coordinates and zero value columns stay zero through the update).
// One CTA of 256 threads per (sequence, value head): threads v and v + 128 hold the two 64-row halves of
// column v of h in fp32 registers, so u and o are dot products inside a thread plus one sum of two
// halves, and every state row moves as one coalesced 512-byte access per half-block of threads (the
// [V][K] layout: one contiguous 256-byte half column per thread).  The kernel is bound by HBM: 64 KB of
// state read and 64 KB written per (sequence, head), plus 1 KB of token data per token.
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace gdr {
namespace {

constexpr int DN = 128;  // the largest head dim: one thread per value column, one key row per state element

struct DecArgs {
    const void *q, *k, *v, *g, *beta;
    const float *state_in;  // nullable: zero start
    float *state_out;       // may alias state_in
    void *o;
    int B, T, Hq, Hv;
    int K, V;  // head dims (<= 128): threads v >= V and state rows d >= K carry zeros
    float scale;
    bool gate_f32, l2norm, v_first;
    unsigned flags;  // gate / beta activations
};

// Sum over the 256 threads of the block (fixed order: warp butterflies, then the eight warp sums).
__device__ __forceinline__ float block_sum(float x, float *red, int lane, int warp) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0) red[warp] = x;
    __syncthreads();
    const float s = ((red[0] + red[1]) + (red[2] + red[3])) + ((red[4] + red[5]) + (red[6] + red[7]));
    __syncthreads();
    return s;
}

// Two threads per value column: thread t holds rows 64 (t / 128) .. +63 of column t % 128 (64 registers, so
// two CTAs of eight warps fit on an SM), and the two halves of each dot product meet in shared memory.
// FULL: K = V = 128 (every mask below is compile-time true); otherwise the masks of smaller head dims.
template <typename T, bool FULL>
__global__ void __launch_bounds__(2 * DN) decode_kernel(const DecArgs a) {
    constexpr int HR = DN / 2;  // state rows per thread
    __shared__ __align__(16) float sq[DN];
    __shared__ __align__(16) float sk[DN];
    __shared__ float pu[2][DN], po[2][DN];  // the two halves' partial dot products
    __shared__ float red[8];
    // one flat grid dimension (x allows 2^31 - 1 blocks): block b = (row n, value head j)
    const int j = (int)(blockIdx.x % (unsigned)a.Hv), n = (int)(blockIdx.x / (unsigned)a.Hv), tid = threadIdx.x;
    const int v = tid & (DN - 1), half = tid >> 7, d0 = half * HR;
    const int lane = tid & 31, warp = tid >> 5;
    const int hq = j / (a.Hv / a.Hq);
    const int K = FULL ? DN : a.K, V = FULL ? DN : a.V;
    const bool vc = FULL || v < V;  // this thread's value column exists
    const size_t sbase = ((size_t)n * a.Hv + j) * K * V;

    float h[HR];  // h[i] = h_{d0+i, v} (zero for rows d0+i >= K or columns v >= V)
    if (a.state_in) {
        if (a.v_first) {
            const float4 *col = reinterpret_cast<const float4 *>(a.state_in + sbase + (size_t)v * K + d0);
#pragma unroll
            for (int i = 0; i < HR / 4; ++i) {
                const float4 x = (vc && (FULL || d0 + 4 * i < K)) ? col[i] : make_float4(0.f, 0.f, 0.f, 0.f);
                h[4 * i] = x.x, h[4 * i + 1] = x.y, h[4 * i + 2] = x.z, h[4 * i + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < HR; ++i)
                h[i] = (vc && (FULL || d0 + i < K)) ? a.state_in[sbase + (size_t)(d0 + i) * V + v] : 0.f;
        }
    } else {
#pragma unroll
        for (int i = 0; i < HR; ++i) h[i] = 0.f;
    }

    const T *q = static_cast<const T *>(a.q);
    const T *k = static_cast<const T *>(a.k);
    const T *vv = static_cast<const T *>(a.v);
    T *o = static_cast<T *>(a.o);
    for (int t = 0; t < a.T; ++t) {
        const long long tk = ((long long)n * a.T + t) * a.Hq + hq;  // token row of q, k
        const long long tv = ((long long)n * a.T + t) * a.Hv + j;   // token row of v, g, beta, o
        // the first half's threads bring q and k (element v); both halves need v, g and beta
        const float qe = (half == 0 && (FULL || v < K)) ? Elt<T>::to_f(q[tk * K + v]) : 0.f;
        const float ke = (half == 0 && (FULL || v < K)) ? Elt<T>::to_f(k[tk * K + v]) : 0.f;
        const float ve = vc ? Elt<T>::to_f(vv[tv * V + v]) : 0.f;
        const float gt = gate_of(load_gate<T>(a.g, tv, a.gate_f32), a.flags);
        const float bt = beta_of(load_gate<T>(a.beta, tv, a.gate_f32), a.flags);
        float rq = 1.f, rk = 1.f;
        if (a.l2norm) {
            rq = 1.0f / sqrtf(block_sum(qe * qe, red, lane, warp) + L2_EPS);
            rk = 1.0f / sqrtf(block_sum(ke * ke, red, lane, warp) + L2_EPS);
        }
        if (half == 0) {
            sq[v] = qe * rq;
            sk[v] = ke * rk;
        }
        __syncthreads();
        const float4 *k4 = reinterpret_cast<const float4 *>(sk + d0);
        const float4 *q4 = reinterpret_cast<const float4 *>(sq + d0);
        float u = 0.f;
#pragma unroll
        for (int i = 0; i < HR / 4; ++i) {
            const float4 kk = k4[i];
            u = fmaf(h[4 * i], kk.x, u);
            u = fmaf(h[4 * i + 1], kk.y, u);
            u = fmaf(h[4 * i + 2], kk.z, u);
            u = fmaf(h[4 * i + 3], kk.w, u);
        }
        pu[half][v] = u;
        __syncthreads();
        u = pu[0][v] + pu[1][v];  // h^T k, both halves in a fixed order
        const float e = __expf(gt);
        const float w = bt * (ve - e * u);
        float ov = 0.f;
#pragma unroll
        for (int i = 0; i < HR / 4; ++i) {
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
        po[half][v] = ov;
        __syncthreads();
        if (half == 0 && vc) o[tv * V + v] = Elt<T>::from_f(a.scale * (po[0][v] + po[1][v]));
        __syncthreads();  // sq, sk, pu, po are rewritten by the next token
    }

    if (!vc) return;
    if (a.v_first) {
        float4 *col = reinterpret_cast<float4 *>(a.state_out + sbase + (size_t)v * K + d0);
#pragma unroll
        for (int i = 0; i < HR / 4; ++i)
            if (FULL || d0 + 4 * i < K) col[i] = make_float4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
    } else {
#pragma unroll
        for (int i = 0; i < HR; ++i)
            if (FULL || d0 + i < K) a.state_out[sbase + (size_t)(d0 + i) * V + v] = h[i];
    }
}

template <typename T>
cudaError_t decode_t(const DecArgs &d, cudaStream_t s) {
    if (d.B == 0) return cudaSuccess;
    const dim3 grid((unsigned)((long long)d.Hv * d.B));
    if (d.K == DN && d.V == DN) return launch_plain(decode_kernel<T, true>, grid, dim3(2 * DN), 0, s, d);
    return launch_plain(decode_kernel<T, false>, grid, dim3(2 * DN), 0, s, d);
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
    d.K = a.K;
    d.V = a.V;
    d.scale = a.scale;
    d.gate_f32 = a.gate_f32;
    d.l2norm = a.l2norm;
    d.v_first = a.v_first;
    d.flags = a.flags;
    return a.bf16 ? decode_t<__nv_bfloat16>(d, s) : decode_t<__half>(d, s);
}

}  // namespace gdr
