// Backward kernels of the chunked gated delta rule.
//
// Per chunk c (C = 64 tokens, G the chunk-local cumsum of g, Gl = G at the
// last valid row, K~ = diag(e^{Gl - G}) K, P = (Q K^T) o Gamma o M), with the
// forward's W = A diag(beta e^G) K, U = A diag(beta) V, Delta = U - W h_c and
// dH' the gradient arriving at the state after the chunk:
//
//   chain_bwd   one CTA per (sequence, value head, value tile), chunks in
//               reverse order, the fp32 state gradient in registers:
//                   dDelta = K~ dH' + scale P^T dO
//                   dH     = e^{Gl} dH' + scale (diag(e^G) Q)^T dO - W^T dDelta
//               and it stores every chunk's dH' for bwd_chunk; dh0 is the last dH.
//   bwd_chunk   one CTA per (chunk, q/k head), visiting the value heads of its
//               group in order; all remaining gradients of the chunk:
//                   dQ = scale diag(e^G) dO h^T + dS K,     dS = (scale dO Delta^T) o Gamma o M
//                   dK = dS^T Q + diag(e^{Gl-G}) Delta dH'^T + diag(beta e^G) A^T dW + dKK K + dKK^T K
//                   dW = -dDelta h^T,  dA = dW (diag(beta e^G) K)^T + dDelta (diag(beta) V)^T
//                   dL = -A^T dA A^T (strictly lower),  dKK = dL o beta_r Gamma
//                   dV = diag(beta) A^T dDelta,  dbeta, dG (then dg = reverse cumsum of dG)
//               followed by the L2-norm chain rule and the group sum for q/k.
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace gdr {

constexpr int VT = 64;

__device__ __forceinline__ void cp_async4b(uint32_t dst, const void *src, bool valid) {
    const int n = valid ? 4 : 0;
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}

template <typename T>
__device__ __forceinline__ void scale_cols2(uint32_t *dst, const uint32_t *src, const float *sB, const float *sG,
                                            bool with_g, int k0, int tq) {
    const int c = k0 + tq * 2;
    float f[4];
    const int cc[4] = {c, c + 1, c + 8, c + 9};
#pragma unroll
    for (int u = 0; u < 4; ++u) f[u] = with_g ? sB[cc[u]] * __expf(sG[cc[u]]) : sB[cc[u]];
    float2 x;
    x = Elt<T>::unpack(src[0]);
    dst[0] = Elt<T>::pack(x.x * f[0], x.y * f[1]);
    x = Elt<T>::unpack(src[1]);
    dst[1] = Elt<T>::pack(x.x * f[0], x.y * f[1]);
    x = Elt<T>::unpack(src[2]);
    dst[2] = Elt<T>::pack(x.x * f[2], x.y * f[3]);
    x = Elt<T>::unpack(src[3]);
    dst[3] = Elt<T>::pack(x.x * f[2], x.y * f[3]);
}

// ============================================================================ chain_bwd

struct ChainBwdP {
    const void *q, *k, *A, *beta, *dout;
    const float *g_cs, *dht;
    void *dhn;     // [rows,Hv,K,V] dtype: gradient w.r.t. the state after each chunk
    float *dh0;
    bool gate_f32, l2norm, v_first;
    float scale;
};

constexpr int CB_Q = 0, CB_K = C * DK * 2, CB_A = 2 * C * DK * 2, CB_DO = CB_A + C * C * 2, CB_G = CB_DO + C * VT * 2,
              CB_B = CB_G + C * 4, CB_STAGE = CB_B + C * 4;
constexpr int CB_DH = 2 * CB_STAGE, CB_W = CB_DH + DK * VT * 2, CB_DD = CB_W + C * DK * 2, CB_DOG = CB_DD + C * VT * 2,
              CB_SMEM = CB_DOG + C * VT * 2;

template <typename T>
__global__ void __launch_bounds__(128, 1) chain_bwd_kernel(Geo geo, ChainBwdP p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const int vt = blockIdx.x, j = blockIdx.y, n = blockIdx.z;
    const int Hv = geo.Hv, Hq = geo.Hq, hq = j / (Hv / Hq);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, tq = lane & 3;
    long long tok0;
    int len, row0;
    geo.seq(n, tok0, len, row0);
    const int nc = (len + C - 1) / C;
    const T *q = static_cast<const T *>(p.q);
    const T *k = static_cast<const T *>(p.k);
    const T *A = static_cast<const T *>(p.A);
    const T *dout = static_cast<const T *>(p.dout);
    const long long st_base = ((long long)n * Hv + j) * DK * DV;

    float dh[2][8][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int d = warp * 32 + mt * 16 + gq + (e >> 1) * 8;
                const int col = vt * VT + nt * 8 + tq * 2 + (e & 1);
                float x = 0.f;
                if (p.dht) x = p.dht[st_base + (p.v_first ? (long long)col * DK + d : (long long)d * DV + col)];
                dh[mt][nt][e] = x;
            }

    float breg = 0.f;
    auto prefetch = [&](int i) {
        unsigned char *sb = smem + (i & 1) * CB_STAGE;
        const long long tb = tok0 + (long long)i * C;
        const int valid = min(C, len - i * C);
        load_rows_async<T>(make_tile(sb + CB_Q, DK), q + (tb * Hq + hq) * DK, (long long)Hq * DK, C, valid, DK, tid,
                           128);
        load_rows_async<T>(make_tile(sb + CB_K, DK), k + (tb * Hq + hq) * DK, (long long)Hq * DK, C, valid, DK, tid,
                           128);
        load_rows_async<T>(make_tile(sb + CB_A, C), A + (tb * Hv + j) * C, (long long)Hv * C, C, valid, C, tid, 128);
        load_rows_async<T>(make_tile(sb + CB_DO, VT), dout + (tb * Hv + j) * DV + vt * VT, (long long)Hv * DV, C,
                           valid, VT, tid, 128);
        if (tid < C) {
            const bool ok = tid < valid;
            cp_async4b(smem_u32(sb + CB_G) + tid * 4, p.g_cs + (ok ? (tb + tid) * Hv + j : 0), ok);
            breg = ok ? load_gate<T>(p.beta, (tb + tid) * Hv + j, p.gate_f32) : 0.f;
        }
        cp_async_commit();
    };
    if (nc > 0) prefetch(nc - 1);

    const Tile tdh = make_tile(smem + CB_DH, VT), tW = make_tile(smem + CB_W, DK);
    const Tile tdD = make_tile(smem + CB_DD, VT), tdOg = make_tile(smem + CB_DOG, VT);
    for (int i = nc - 1; i >= 0; --i) {
        unsigned char *sb = smem + (i & 1) * CB_STAGE;
        float *sG = reinterpret_cast<float *>(sb + CB_G);
        float *sB = reinterpret_cast<float *>(sb + CB_B);
        cp_async_wait<0>();
        if (tid < C) sB[tid] = breg;
        // gradient w.r.t. the state after this chunk: bf16 copy for the MMAs and for bwd_chunk
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) store_acc<T, 8>(tdh, dh[mt], warp * 32 + mt * 16, 0, lane);
        {
            T *o = static_cast<T *>(p.dhn);
            const long long hb = ((long long)(row0 + i) * Hv + j) * DK * DV;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int d = warp * 32 + mt * 16 + gq + hh * 8;
                        const int col = vt * VT + nt * 8 + tq * 2;
                        *reinterpret_cast<uint32_t *>(o + hb + (long long)d * DV + col) =
                            Elt<T>::pack(dh[mt][nt][2 * hh], dh[mt][nt][2 * hh + 1]);
                    }
        }
        __syncthreads();
        const Tile tqk = make_tile(sb + CB_Q, DK), tkk = make_tile(sb + CB_K, DK);
        const Tile ta = make_tile(sb + CB_A, C), tdo = make_tile(sb + CB_DO, VT);
        const int valid = min(C, len - i * C);
        if (p.l2norm) {
            l2norm_rows<T>(tqk, valid, warp, 4, lane);
            l2norm_rows<T>(tkk, valid, warp, 4, lane);
            __syncthreads();
        }
        if (i > 0) prefetch(i - 1);
        const float Gl = sG[valid - 1];
        const int r0 = warp * 16;

        // ---- W rows r0.. -> shared (for W^T dDelta)
        {
            uint32_t aw[4][4];
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                uint32_t a[4];
                load_a(a, ta, r0, ks * 16, false, lane);
                scale_cols2<T>(aw[ks], a, sB, sG, true, ks * 16, tq);
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float wacc[8][4];
                zero_acc<8>(wacc);
                warp_mma_ra<T, 8, 4>(wacc, aw, tkk, half * 64, true, 0, lane);
                store_acc<T, 8>(tW, wacc, r0, half * 64, lane);
            }
        }
        // ---- scale diag(e^G) dO rows r0.. -> shared
        {
            const float e0 = p.scale * __expf(sG[r0 + gq]), e1 = p.scale * __expf(sG[r0 + gq + 8]);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const int col = nt * 8 + tq * 2;
                const float2 x0 = Elt<T>::unpack(lds32(tdo.addr(r0 + gq, col)));
                const float2 x1 = Elt<T>::unpack(lds32(tdo.addr(r0 + gq + 8, col)));
                sts32(tdOg.addr(r0 + gq, col), Elt<T>::pack(x0.x * e0, x0.y * e0));
                sts32(tdOg.addr(r0 + gq + 8, col), Elt<T>::pack(x1.x * e1, x1.y * e1));
            }
        }
        // ---- dDelta rows r0.. = e^{Gl-G_r} (K dH')_r + scale (P^T dO)_r ; stored negated
        {
            float acc[8][4];
            zero_acc<8>(acc);
            warp_mma<T, 8, 8>(acc, tkk, r0, false, tdh, 0, true, 0, lane);
            const float f0 = __expf(Gl - sG[r0 + gq]), f1 = __expf(Gl - sG[r0 + gq + 8]);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                acc[nt][0] *= f0;
                acc[nt][1] *= f0;
                acc[nt][2] *= f1;
                acc[nt][3] *= f1;
            }
            // P^T rows r: (k_r . q_s) e^{G_s - G_r} for valid s >= r
            float pacc[8][4];
            zero_acc<8>(pacc);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                uint32_t a[4];
                load_a(a, tkk, r0, ks * 16, false, lane);
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    if (np >= warp) {
                        uint32_t b[4];
                        load_b2(b, tqk, np * 16, ks * 16, false, lane);
                        mma16816<T>(pacc[2 * np], a, b[0], b[1]);
                        mma16816<T>(pacc[2 * np + 1], a, b[2], b[3]);
                    }
                }
            }
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = r0 + gq + (e >> 1) * 8, s = nt * 8 + tq * 2 + (e & 1);
                    pacc[nt][e] = (s >= r && s < valid) ? pacc[nt][e] * p.scale * __expf(sG[s] - sG[r]) : 0.f;
                }
            uint32_t pt[4][4];
            acc_to_a<T, 4>(pt, pacc);
            warp_mma_ra<T, 8, 4>(acc, pt, tdo, 0, true, 0, lane);
            store_acc<T, 8>(tdD, acc, r0, 0, lane, -1.f);
        }
        __syncthreads();

        // ---- dH = e^{Gl} dH' + Q^T (scale e^G dO) - W^T dDelta
        {
            const float eg = __expf(Gl);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
                for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) dh[mt][nt][e] *= eg;
                warp_mma<T, 8, 4>(dh[mt], tqk, warp * 32 + mt * 16, true, tdOg, 0, true, 0, lane);
                warp_mma<T, 8, 4>(dh[mt], tW, warp * 32 + mt * 16, true, tdD, 0, true, 0, lane);
            }
        }
        __syncthreads();
    }

    if (p.dh0) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int d = warp * 32 + mt * 16 + gq + (e >> 1) * 8;
                    const int col = vt * VT + nt * 8 + tq * 2 + (e & 1);
                    p.dh0[st_base + (p.v_first ? (long long)col * DK + d : (long long)d * DV + col)] = dh[mt][nt][e];
                }
    }
}

template <typename T>
static cudaError_t chain_bwd_t(const Args &a, const ChainBwdP &p, cudaStream_t s) {
    auto kern = chain_bwd_kernel<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, CB_SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(DV / VT, a.Hv, a.N);
    kern<<<grid, 128, CB_SMEM, s>>>(make_geo(a), p);
    return cudaGetLastError();
}

cudaError_t launch_chain_bwd(const Args &a, const void *q, const void *k, const float *g_cs, const void *beta,
                             const void *A, const void *dout, const float *dht, void *dhn, float *dh0,
                             cudaStream_t s) {
    ChainBwdP p;
    p.q = q;
    p.k = k;
    p.A = A;
    p.beta = beta;
    p.dout = dout;
    p.g_cs = g_cs;
    p.dht = dht;
    p.dhn = dhn;
    p.dh0 = dh0;
    p.gate_f32 = a.gate_f32;
    p.l2norm = a.l2norm;
    p.v_first = a.v_first;
    p.scale = a.scale;
    return a.bf16 ? chain_bwd_t<__nv_bfloat16>(a, p, s) : chain_bwd_t<__half>(a, p, s);
}

// ============================================================================ bwd_chunk

#include "bwd_chunk.cuh"

}  // namespace gdr
