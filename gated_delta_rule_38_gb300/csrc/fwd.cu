// Forward kernels of the chunked gated delta rule.
//
//   wy_fwd     one CTA per (chunk, value head): chunk-local cumsum of the
//              log-gate, L = strictly-lower(diag(beta) (K K^T o exp(G_r - G_s))),
//              A = (I + L)^-1 (16x16 diagonal blocks by substitution in fp32,
//              off-diagonal blocks merged with tf32 tensor-core products).
//   chain_fwd  one CTA per (sequence, value head, 64-column value tile): walks
//              the chunks in order with the fp32 state in registers:
//                  W = A diag(beta e^G) K,  U = A diag(beta) V,  Delta = U - W h
//                  O = scale (diag(e^G) Q h + (Q K^T o Gamma o M) Delta)
//                  h <- e^{G_last} h + K^T diag(e^{G_last - G}) Delta
//              These are the chunk form of the token recurrence
//              S_t = e^{g_t} S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T.
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace gdr {

// ============================================================================ wy_fwd

constexpr int LDF = 68;  // fp32 row stride of the 64x64 matrices (bank spread)
constexpr int WY_SMEM = C * DK * 2 + 2 * C * LDF * 4 + 2 * C * 4 + 4 * 16 * 20 * 4;

template <typename T>
__global__ void __launch_bounds__(128) wy_fwd_kernel(Geo geo, const T *__restrict__ k, const void *__restrict__ g,
                                                     const void *__restrict__ beta, bool gate_f32, bool l2norm,
                                                     float *__restrict__ g_cs, T *__restrict__ A_out) {
    extern __shared__ __align__(1024) unsigned char smem[];
    T *sk = reinterpret_cast<T *>(smem);
    float *Lm = reinterpret_cast<float *>(smem + C * DK * 2);
    float *Ai = Lm + C * LDF;
    float *sG = Ai + C * LDF;
    float *sB = sG + C;
    float *scr = sB + C;  // [4 warps][16][20]

    long long tok0;
    int len, n, ci;
    if (!geo.chunk(blockIdx.x, tok0, len, n, ci)) return;
    const int j = blockIdx.y, Hv = geo.Hv, Hq = geo.Hq;
    const int hq = j / (Hv / Hq);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, tq = lane & 3;

    const Tile tk = make_tile(sk, DK);
    load_rows_async<T>(tk, k + (tok0 * Hq + hq) * DK, (long long)Hq * DK, C, len, DK, tid, 128);
    cp_async_commit();
    if (tid < C) {
        float gv = 0.f, bv = 0.f;
        if (tid < len) {
            gv = load_gate<T>(g, (tok0 + tid) * Hv + j, gate_f32);
            bv = load_gate<T>(beta, (tok0 + tid) * Hv + j, gate_f32);
        }
        sG[tid] = gv;
        sB[tid] = bv;
    }
    cp_async_wait<0>();
    __syncthreads();
    if (l2norm) l2norm_rows<T>(tk, len, warp, 4, lane);
    if (warp == 0) {
        float x0 = sG[lane], x1 = sG[lane + 32];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y0 = __shfl_up_sync(0xffffffffu, x0, o);
            const float y1 = __shfl_up_sync(0xffffffffu, x1, o);
            if (lane >= o) {
                x0 += y0;
                x1 += y1;
            }
        }
        x1 += __shfl_sync(0xffffffffu, x0, 31);
        sG[lane] = x0;
        sG[lane + 32] = x1;
        if (lane < len) g_cs[(tok0 + lane) * Hv + j] = x0;
        if (lane + 32 < len) g_cs[(tok0 + lane + 32) * Hv + j] = x1;
    }
    __syncthreads();

    // ---- L (warp w owns rows 16w..16w+15; only column tiles at or left of the diagonal)
    {
        float acc[8][4];
        zero_acc<8>(acc);
        const int r0 = warp * 16;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t a[4];
            load_a(a, tk, r0, ks * 16, false, lane);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                if (np <= warp) {
                    uint32_t b[4];
                    load_b2(b, tk, np * 16, ks * 16, false, lane);
                    mma16816<T>(acc[2 * np], a, b[0], b[1]);
                    mma16816<T>(acc[2 * np + 1], a, b[2], b[3]);
                }
            }
        }
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = r0 + gq + 8 * hh;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int s = nt * 8 + tq * 2 + e;
                    float val = 0.f;
                    if (s < r && r < len) val = sB[r] * __expf(sG[r] - sG[s]) * acc[nt][2 * hh + e];
                    Lm[r * LDF + s] = val;
                }
            }
    }
    __syncthreads();

    // ---- diagonal 16x16 blocks: warp w, lane c < 16 solves column c of (I + L_ww)^-1
    if (lane < 16) {
        const int b0 = warp * 16;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float acc = 0.f;
#pragma unroll
            for (int s = 0; s < i; ++s) acc += Lm[(b0 + i) * LDF + b0 + s] * x[s];
            x[i] = (i == lane) ? 1.f : (i > lane ? -acc : 0.f);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) Ai[(b0 + i) * LDF + b0 + lane] = x[i];
    }
    __syncthreads();

    // ---- off-diagonal blocks, one block row at a time:
    //      A_ij = -A_ii * sum_{k=j}^{i-1} L_ik A_kj
    float *ws = scr + warp * 16 * 20;
    for (int bi = 1; bi < 4; ++bi) {
        if (warp < bi) {
            const int bj = warp;
            float r[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            for (int kb = bj; kb < bi; ++kb) {
#pragma unroll
                for (int k8 = 0; k8 < 2; ++k8) {
                    const int kc = kb * 16 + k8 * 8;
                    uint32_t a[4];
                    a[0] = to_tf32(Lm[(bi * 16 + gq) * LDF + kc + tq]);
                    a[1] = to_tf32(Lm[(bi * 16 + gq + 8) * LDF + kc + tq]);
                    a[2] = to_tf32(Lm[(bi * 16 + gq) * LDF + kc + tq + 4]);
                    a[3] = to_tf32(Lm[(bi * 16 + gq + 8) * LDF + kc + tq + 4]);
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const uint32_t b0 = to_tf32(Ai[(kc + tq) * LDF + bj * 16 + nt * 8 + gq]);
                        const uint32_t b1 = to_tf32(Ai[(kc + tq + 4) * LDF + bj * 16 + nt * 8 + gq]);
                        mma1688_tf32(r[nt], a, b0, b1);
                    }
                }
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                ws[gq * 20 + nt * 8 + tq * 2] = r[nt][0];
                ws[gq * 20 + nt * 8 + tq * 2 + 1] = r[nt][1];
                ws[(gq + 8) * 20 + nt * 8 + tq * 2] = r[nt][2];
                ws[(gq + 8) * 20 + nt * 8 + tq * 2 + 1] = r[nt][3];
            }
            __syncwarp();
            float o[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int k8 = 0; k8 < 2; ++k8) {
                const int kc = bi * 16 + k8 * 8;
                uint32_t a[4];
                a[0] = to_tf32(Ai[(bi * 16 + gq) * LDF + kc + tq]);
                a[1] = to_tf32(Ai[(bi * 16 + gq + 8) * LDF + kc + tq]);
                a[2] = to_tf32(Ai[(bi * 16 + gq) * LDF + kc + tq + 4]);
                a[3] = to_tf32(Ai[(bi * 16 + gq + 8) * LDF + kc + tq + 4]);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const uint32_t b0 = to_tf32(ws[(k8 * 8 + tq) * 20 + nt * 8 + gq]);
                    const uint32_t b1 = to_tf32(ws[(k8 * 8 + tq + 4) * 20 + nt * 8 + gq]);
                    mma1688_tf32(o[nt], a, b0, b1);
                }
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int c = bj * 16 + nt * 8 + tq * 2;
                Ai[(bi * 16 + gq) * LDF + c] = -o[nt][0];
                Ai[(bi * 16 + gq) * LDF + c + 1] = -o[nt][1];
                Ai[(bi * 16 + gq + 8) * LDF + c] = -o[nt][2];
                Ai[(bi * 16 + gq + 8) * LDF + c + 1] = -o[nt][3];
            }
            __syncwarp();
        }
        __syncthreads();
    }

    // ---- A out: row r of the chunk at token tok0 + r, zero above the diagonal
    for (int i = tid; i < C * 8; i += 128) {
        const int r = i >> 3, c0 = (i & 7) * 8;
        if (r >= len) continue;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = c0 + 2 * e;
            const float lo = (c <= r) ? Ai[r * LDF + c] : 0.f;
            const float hi = (c + 1 <= r) ? Ai[r * LDF + c + 1] : 0.f;
            w[e] = Elt<T>::pack(lo, hi);
        }
        *reinterpret_cast<uint4 *>(A_out + ((tok0 + r) * Hv + j) * C + c0) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// ============================================================================ chain_fwd

struct FwdP {
    const void *q, *k, *v, *A, *beta;
    const float *g_cs, *h0;
    void *o, *h;
    float *fin;
    bool gate_f32, l2norm, v_first, h_api;
    float scale;
};

constexpr int VT = 64;  // value columns per CTA
// shared-memory layout of chain_fwd (bytes)
constexpr int CF_Q = 0, CF_K = C * DK * 2, CF_V = 2 * C * DK * 2, CF_A = CF_V + C * VT * 2, CF_G = CF_A + C * C * 2,
              CF_B = CF_G + C * 4, CF_STAGE = CF_B + C * 4;
constexpr int CF_H = 2 * CF_STAGE, CF_D = CF_H + 2 * DK * VT * 2, CF_DT = CF_D + C * VT * 2,
              CF_SMEM = CF_DT + C * VT * 2;

__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, bool valid) {
    const int n = valid ? 4 : 0;
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}

// Scale the columns of a 16x16 A fragment held as packed pairs: column c of
// the k-step is multiplied by beta[c] (times e^{G[c]} when with_g).
template <typename T>
__device__ __forceinline__ void scale_cols(uint32_t *dst, const uint32_t *src, const float *sB, const float *sG,
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

template <typename T, bool WRITE_O>
__global__ void __launch_bounds__(128, 1) chain_fwd_kernel(Geo geo, FwdP p) {
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
    const T *v = static_cast<const T *>(p.v);
    const T *A = static_cast<const T *>(p.A);
    const long long st_base = ((long long)n * Hv + j) * DK * DV;

    // fp32 state: warp w owns key rows 32w..32w+31 of this CTA's value tile
    float hacc[2][8][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int d = warp * 32 + mt * 16 + gq + (e >> 1) * 8;
                const int col = vt * VT + nt * 8 + tq * 2 + (e & 1);
                float x = 0.f;
                if (p.h0) x = p.h0[st_base + (p.v_first ? (long long)col * DK + d : (long long)d * DV + col)];
                hacc[mt][nt][e] = x;
            }

    auto sh_tile = [&](int b) { return make_tile(smem + CF_H + b * DK * VT * 2, VT); };
    auto write_state = [&](const Tile &t) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) store_acc<T, 8>(t, hacc[mt], warp * 32 + mt * 16, 0, lane);
    };
    write_state(sh_tile(0));

    float breg = 0.f;
    auto prefetch = [&](int i) {
        unsigned char *sb = smem + (i & 1) * CF_STAGE;
        const long long tb = tok0 + (long long)i * C;
        const int valid = min(C, len - i * C);
        if (WRITE_O)
            load_rows_async<T>(make_tile(sb + CF_Q, DK), q + (tb * Hq + hq) * DK, (long long)Hq * DK, C, valid, DK,
                               tid, 128);
        load_rows_async<T>(make_tile(sb + CF_K, DK), k + (tb * Hq + hq) * DK, (long long)Hq * DK, C, valid, DK, tid,
                           128);
        load_rows_async<T>(make_tile(sb + CF_V, VT), v + (tb * Hv + j) * DV + vt * VT, (long long)Hv * DV, C, valid,
                           VT, tid, 128);
        load_rows_async<T>(make_tile(sb + CF_A, C), A + (tb * Hv + j) * C, (long long)Hv * C, C, valid, C, tid, 128);
        if (tid < C) {
            const bool ok = tid < valid;
            cp_async4(smem_u32(sb + CF_G) + tid * 4, p.g_cs + (ok ? (tb + tid) * Hv + j : 0), ok);
            breg = ok ? load_gate<T>(p.beta, (tb + tid) * Hv + j, p.gate_f32) : 0.f;
        }
        cp_async_commit();
    };
    if (nc > 0) prefetch(0);

    for (int i = 0; i < nc; ++i) {
        unsigned char *sb = smem + (i & 1) * CF_STAGE;
        float *sG = reinterpret_cast<float *>(sb + CF_G);
        float *sB = reinterpret_cast<float *>(sb + CF_B);
        cp_async_wait<0>();
        if (tid < C) sB[tid] = breg;
        __syncthreads();
        const Tile tqk = make_tile(sb + CF_Q, DK), tkk = make_tile(sb + CF_K, DK);
        const Tile tv = make_tile(sb + CF_V, VT), ta = make_tile(sb + CF_A, C);
        const Tile hcur = sh_tile(i & 1), hnext = sh_tile((i + 1) & 1);
        const Tile tD = make_tile(smem + CF_D, VT), tDt = make_tile(smem + CF_DT, VT);
        const int valid = min(C, len - i * C);
        if (p.l2norm) {
            if (WRITE_O) l2norm_rows<T>(tqk, valid, warp, 4, lane);
            l2norm_rows<T>(tkk, valid, warp, 4, lane);
            __syncthreads();
        }
        if (i + 1 < nc) prefetch(i + 1);
        const float Gl = sG[valid - 1];
        const int r0 = warp * 16;

        // ---- Delta = A diag(beta) V - A diag(beta e^G) K h   (rows r0..r0+15)
        float dacc[8][4];
        {
            uint32_t af[4][4], aw[4][4];
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                uint32_t a[4];
                load_a(a, ta, r0, ks * 16, false, lane);
                scale_cols<T>(af[ks], a, sB, sG, false, ks * 16, tq);
                scale_cols<T>(aw[ks], a, sB, sG, true, ks * 16, tq);
            }
            zero_acc<8>(dacc);
            warp_mma_ra<T, 8, 4>(dacc, af, tv, 0, true, 0, lane);  // U
            uint32_t wf[8][4];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float wacc[8][4];
                zero_acc<8>(wacc);
                warp_mma_ra<T, 8, 4>(wacc, aw, tkk, half * 64, true, 0, lane);
                acc_to_a<T, 4>(&wf[half * 4], wacc, -1.f);
            }
            warp_mma_ra<T, 8, 8>(dacc, wf, hcur, 0, true, 0, lane);  // U - W h
        }
        store_acc<T, 8>(tD, dacc, r0, 0, lane);
        {
            const float f0 = __expf(Gl - sG[r0 + gq]), f1 = __expf(Gl - sG[r0 + gq + 8]);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const int col = nt * 8 + tq * 2;
                sts32(tDt.addr(r0 + gq, col), Elt<T>::pack(dacc[nt][0] * f0, dacc[nt][1] * f0));
                sts32(tDt.addr(r0 + gq + 8, col), Elt<T>::pack(dacc[nt][2] * f1, dacc[nt][3] * f1));
            }
        }
        __syncthreads();

        // ---- O = scale (diag(e^G) Q h + P Delta)
        if (WRITE_O) {
            uint32_t pf[4][4];
            {
                float pacc[8][4];
                zero_acc<8>(pacc);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    uint32_t a[4];
                    load_a(a, tqk, r0, ks * 16, false, lane);
#pragma unroll
                    for (int np = 0; np < 4; ++np) {
                        if (np <= warp) {
                            uint32_t b[4];
                            load_b2(b, tkk, np * 16, ks * 16, false, lane);
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
                        pacc[nt][e] = (s <= r && r < valid) ? pacc[nt][e] * __expf(sG[r] - sG[s]) : 0.f;
                    }
                acc_to_a<T, 4>(pf, pacc);
            }
            float oacc[8][4];
            zero_acc<8>(oacc);
            warp_mma<T, 8, 8>(oacc, tqk, r0, false, hcur, 0, true, 0, lane);
            const float e0 = __expf(sG[r0 + gq]), e1 = __expf(sG[r0 + gq + 8]);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                oacc[nt][0] *= e0;
                oacc[nt][1] *= e0;
                oacc[nt][2] *= e1;
                oacc[nt][3] *= e1;
            }
            warp_mma_ra<T, 8, 4>(oacc, pf, tD, 0, true, 0, lane);
            T *o = static_cast<T *>(p.o);
            const long long tb = tok0 + (long long)i * C;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = r0 + gq + hh * 8;
                if (r < valid) {
                    T *orow = o + ((tb + r) * Hv + j) * DV + vt * VT;
#pragma unroll
                    for (int nt = 0; nt < 8; ++nt)
                        *reinterpret_cast<uint32_t *>(orow + nt * 8 + tq * 2) =
                            Elt<T>::pack(oacc[nt][2 * hh] * p.scale, oacc[nt][2 * hh + 1] * p.scale);
                }
            }
        }

        // ---- state before this chunk (optional output)
        if (p.h) {
            T *h = static_cast<T *>(p.h);
            const long long hb = ((long long)(row0 + i) * Hv + j) * DK * DV;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int d = warp * 32 + mt * 16 + gq + hh * 8;
                        const int col = vt * VT + nt * 8 + tq * 2;
                        const float x0 = hacc[mt][nt][2 * hh], x1 = hacc[mt][nt][2 * hh + 1];
                        if (p.h_api && p.v_first) {
                            h[hb + (long long)col * DK + d] = Elt<T>::from_f(x0);
                            h[hb + (long long)(col + 1) * DK + d] = Elt<T>::from_f(x1);
                        } else {
                            *reinterpret_cast<uint32_t *>(h + hb + (long long)d * DV + col) = Elt<T>::pack(x0, x1);
                        }
                    }
        }

        // ---- h <- e^{G_last} h + K^T diag(e^{G_last - G}) Delta
        {
            const float eg = __expf(Gl);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
                for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) hacc[mt][nt][e] *= eg;
                warp_mma<T, 8, 4>(hacc[mt], tkk, warp * 32 + mt * 16, true, tDt, 0, true, 0, lane);
            }
            write_state(hnext);
        }
    }

    if (p.fin) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int d = warp * 32 + mt * 16 + gq + (e >> 1) * 8;
                    const int col = vt * VT + nt * 8 + tq * 2 + (e & 1);
                    p.fin[st_base + (p.v_first ? (long long)col * DK + d : (long long)d * DV + col)] = hacc[mt][nt][e];
                }
    }
}

// ============================================================================ launchers

template <typename T>
static cudaError_t wy_fwd_t(const Args &a, const void *k, const void *g, const void *beta, float *g_cs, void *A,
                            cudaStream_t s) {
    if (a.max_chunks == 0) return cudaSuccess;
    auto kern = wy_fwd_kernel<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, WY_SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)a.max_chunks, a.Hv);
    kern<<<grid, 128, WY_SMEM, s>>>(make_geo(a), static_cast<const T *>(k), g, beta, a.gate_f32, a.l2norm, g_cs,
                                    static_cast<T *>(A));
    return cudaGetLastError();
}

cudaError_t launch_wy_fwd(const Args &a, const void *k, const void *g, const void *beta, float *g_cs, void *A,
                          cudaStream_t s) {
    return a.bf16 ? wy_fwd_t<__nv_bfloat16>(a, k, g, beta, g_cs, A, s) : wy_fwd_t<__half>(a, k, g, beta, g_cs, A, s);
}

template <typename T>
static cudaError_t chain_fwd_t(const Args &a, const FwdP &p, bool write_o, cudaStream_t s) {
    auto kern = write_o ? chain_fwd_kernel<T, true> : chain_fwd_kernel<T, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, CF_SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(DV / VT, a.Hv, a.N);
    kern<<<grid, 128, CF_SMEM, s>>>(make_geo(a), p);
    return cudaGetLastError();
}

cudaError_t launch_chain_fwd(const Args &a, const void *q, const void *k, const void *v, const float *g_cs,
                             const void *beta, const void *A, const float *h0, void *o, float *final_state, void *h,
                             bool h_api_layout, cudaStream_t s) {
    FwdP p;
    p.q = q;
    p.k = k;
    p.v = v;
    p.A = A;
    p.beta = beta;
    p.g_cs = g_cs;
    p.h0 = h0;
    p.o = o;
    p.h = h;
    p.fin = final_state;
    p.gate_f32 = a.gate_f32;
    p.l2norm = a.l2norm;
    p.v_first = a.v_first;
    p.h_api = h_api_layout;
    p.scale = a.scale;
    return a.bf16 ? chain_fwd_t<__nv_bfloat16>(a, p, o != nullptr, s) : chain_fwd_t<__half>(a, p, o != nullptr, s);
}

}  // namespace gdr
