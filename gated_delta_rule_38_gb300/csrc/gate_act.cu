// Gate and beta activations inside the library (the options use_gate_in_kernel, use_beta_sigmoid_in_kernel and
// allow_neg_eigval that the FlashQLA backend's verifier names, PR #998 "[GDN] Add FlashQLA backend dispatch"):
//
//   g    = logsigmoid(x)       with GDR_GATE_IN_KERNEL (x: the raw gate logit; the log of a sigmoid decay)
//   beta = sigmoid(b)          with GDR_BETA_SIGMOID_IN_KERNEL (b: the raw beta)
//   beta = 2 beta              with GDR_ALLOW_NEG_EIGVAL (the eigenvalue 1 - beta along k spans (-1, 1))
//
// The forward activates the raw per-token scalars once into fp32 buffers that the rest of the path reads as
// its gates, and keeps sigmoid(-x) = d logsigmoid(x) / dx for the backward.  The backward activates beta the
// same way, runs on the activated values, and turns the gradients w.r.t. the used g and beta into those w.r.t.
// the raw inputs (chain rule).  All three are elementwise over tokens x value heads: coalesced grid-stride loops.
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace gdr {
namespace {

template <typename T>
__global__ void gate_act_fwd_kernel(const void *g, const void *beta, bool gate_f32, long long n, unsigned flags,
                                    float *geff, float *beff, float *sg) {
    griddep_wait();
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const float x = load_gate<T>(g, i, gate_f32);
        const float b = load_gate<T>(beta, i, gate_f32);
        geff[i] = gate_of(x, flags);
        beff[i] = beta_of(b, flags);
        if (sg) sg[i] = sigmoid_f(-x);
    }
}

template <typename T>
__global__ void gate_act_beta_kernel(const void *beta, bool gate_f32, long long n, unsigned flags, float *beff) {
    griddep_wait();
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        beff[i] = beta_of(load_gate<T>(beta, i, gate_f32), flags);
}

template <typename T>
__global__ void gate_act_bwd_kernel(const float *dgeff, const float *dbeff, const float *sg, const void *beta,
                                    bool gate_f32, long long n, unsigned flags, void *dg, void *dbeta) {
    griddep_wait();
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        float d = dgeff[i];
        if (flags & GDR_GATE_IN_KERNEL) d *= sg[i];
        float e = dbeff[i];
        if (flags & GDR_ALLOW_NEG_EIGVAL) e *= 2.f;
        if (flags & GDR_BETA_SIGMOID_IN_KERNEL) {
            const float s = sigmoid_f(load_gate<T>(beta, i, gate_f32));
            e *= s * (1.f - s);
        }
        store_gate<T>(dg, i, gate_f32, d);
        store_gate<T>(dbeta, i, gate_f32, e);
    }
}

inline unsigned blocks_for(long long n) {
    const long long b = (n + 255) / 256;
    return (unsigned)(b < 4096 ? (b > 0 ? b : 1) : 4096);
}

}  // namespace

cudaError_t launch_gate_act_fwd(const Args &a, const void *g, const void *beta, unsigned flags, float *geff,
                                float *beff, float *sg, cudaStream_t s) {
    const long long n = (long long)a.B * a.T * a.Hv;
    if (n == 0) return cudaSuccess;
    if (a.bf16)
        return launch_plain(gate_act_fwd_kernel<__nv_bfloat16>, dim3(blocks_for(n)), dim3(256), 0, s, g, beta,
                            a.gate_f32, n, flags, geff, beff, sg);
    return launch_plain(gate_act_fwd_kernel<__half>, dim3(blocks_for(n)), dim3(256), 0, s, g, beta, a.gate_f32, n,
                        flags, geff, beff, sg);
}

cudaError_t launch_gate_act_beta(const Args &a, const void *beta, unsigned flags, float *beff, cudaStream_t s) {
    const long long n = (long long)a.B * a.T * a.Hv;
    if (n == 0) return cudaSuccess;
    if (a.bf16)
        return launch_plain(gate_act_beta_kernel<__nv_bfloat16>, dim3(blocks_for(n)), dim3(256), 0, s, beta,
                            a.gate_f32, n, flags, beff);
    return launch_plain(gate_act_beta_kernel<__half>, dim3(blocks_for(n)), dim3(256), 0, s, beta, a.gate_f32, n,
                        flags, beff);
}

cudaError_t launch_gate_act_bwd(const Args &a, const float *dgeff, const float *dbeff, const float *sg,
                                const void *beta, unsigned flags, void *dg, void *dbeta, cudaStream_t s) {
    const long long n = (long long)a.B * a.T * a.Hv;
    if (n == 0) return cudaSuccess;
    if (a.bf16)
        return launch_plain(gate_act_bwd_kernel<__nv_bfloat16>, dim3(blocks_for(n)), dim3(256), 0, s, dgeff, dbeff,
                            sg, beta, a.gate_f32, n, flags, dg, dbeta);
    return launch_plain(gate_act_bwd_kernel<__half>, dim3(blocks_for(n)), dim3(256), 0, s, dgeff, dbeff, sg, beta,
                        a.gate_f32, n, flags, dg, dbeta);
}

}  // namespace gdr
