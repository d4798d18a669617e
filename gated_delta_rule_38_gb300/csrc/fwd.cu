// Forward kernels of the chunked gated delta rule.
//
//   wy_fwd     one CTA per (chunk, value head): chunk-local cumsum of the
//              log-gate, L = strictly-lower(diag(beta) (K K^T o exp(G_r - G_s))),
//              A = (I + L)^-1 (16x16 diagonal blocks by substitution in fp32,
//              off-diagonal blocks merged with tf32 tensor-core products), and the
//              state-independent attention block P = scale (q^ k^T o exp(G_r - G_s)),
//              s <= r, with the inverse q/k norms the recurrence applies as factors.
//              (The backward's P from a given g_cumsum comes from chunk_p_tc.cu.)
// The recurrences that consume A and P live in chain_ws.cu / chain_tc.cu.
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace gdr {

// ============================================================================ wy_fwd

constexpr int LDF = 68;  // fp32 row stride of the 64x64 matrices (bank spread)
constexpr int LDP = C + 8;  // bf16 row stride of the P staging (bank spread)
// [K tile 16 KB][Q tile 16 KB, later L][.. A^-1][gate arrays]; the merge scratch reuses the K tile and the
// P staging the A^-1 buffer, so four CTAs fit on an SM
constexpr int WY_SMEM = C * DK * 2 + 2 * C * LDF * 4 + 4 * C * 4;
static_assert(C * DK * 2 <= C * LDF * 4, "the Q tile must fit under L");

// 1 / sqrt(sum x^2 + eps) of every row r < rows of a [rows x 128] tile (fp32 sums of the stored values);
// each warp takes 8 rows at a time, lane l a quarter (32 values) of row l/4.
template <typename T>
__device__ __forceinline__ void row_inv_norms(const Tile &t, int rows, int warp, int nwarps, int lane, float *inv_out) {
    const int rq = lane >> 2, qq = lane & 3;
    for (int r0 = warp * 8; r0 < rows; r0 += nwarps * 8) {
        const int r = r0 + rq;
        float ss = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint4 u;
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];\n"
                         : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
                         : "r"(t.addr(r, qq * 32 + c * 8)));
            const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 x = Elt<T>::unpack(wv[e]);
                ss = fmaf(x.x, x.x, fmaf(x.y, x.y, ss));
            }
        }
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        if (r < rows && qq == 0) inv_out[r] = 1.0f / sqrtf(ss + L2_EPS);
    }
}

struct WyArgs {
    const void *q, *k, *g, *beta;
    bool gate_f32, l2norm;
    float scale;
    float *g_cs;
    void *A_out;    // [tokens,Hv,64] or nullptr
    void *P_out;    // [tokens,Hv,64]: scale (q^ k^T o Gamma), lower incl. diagonal, or nullptr
    float *rq_out, *rk_out;  // [tokens,Hv] inverse norms (with l2norm), or nullptr
};

template <typename T>
__global__ void __launch_bounds__(128, 4) wy_fwd_kernel(Geo geo, const WyArgs w) {
    griddep_launch_next();
    griddep_wait();
    extern __shared__ __align__(1024) unsigned char smem[];
    T *sk = reinterpret_cast<T *>(smem);
    T *sq = reinterpret_cast<T *>(smem + C * DK * 2);
    float *Lm = reinterpret_cast<float *>(smem + C * DK * 2);  // over the Q tile once P is out
    float *Ai = Lm + C * LDF;
    float *sG = Ai + C * LDF;
    float *sB = sG + C;
    float *sRQ = sB + C;
    float *sRK = sRQ + C;
    float *scr = reinterpret_cast<float *>(smem);  // [4 warps][16][20], over the K tile once L is built
    T *sp = reinterpret_cast<T *>(Ai);             // P staging [64][LDP], before A^-1 is built

    long long tok0;
    int len, n, ci;
    if (!geo.chunk(blockIdx.x, tok0, len, n, ci)) return;
    const int j = blockIdx.y, Hv = geo.Hv, Hq = geo.Hq;
    const int hq = j / (Hv / Hq);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, tq = lane & 3;
    const bool want_p = w.P_out != nullptr;

    const Tile tk = make_tile(sk, DK), tqt = make_tile(sq, DK);
    load_rows_async<T>(tk, static_cast<const T *>(w.k) + (tok0 * Hq + hq) * DK, (long long)Hq * DK, C, len, DK, tid,
                       128);
    if (want_p)
        load_rows_async<T>(tqt, static_cast<const T *>(w.q) + (tok0 * Hq + hq) * DK, (long long)Hq * DK, C, len, DK,
                           tid, 128);
    cp_async_commit();
    if (tid < C) {
        float gv = 0.f, bv = 0.f;
        if (tid < len) {
            gv = load_gate<T>(w.g, (tok0 + tid) * Hv + j, w.gate_f32);
            bv = load_gate<T>(w.beta, (tok0 + tid) * Hv + j, w.gate_f32);
        }
        sG[tid] = gv;
        sB[tid] = bv;
    }
    cp_async_wait<0>();
    __syncthreads();
    // inverse L2 norms of the q and k rows (1 without normalisation): the tiles stay as loaded and the
    // norms enter P and L as row / column factors.  With P they come from the MMA pass's own fragments.
    if (!want_p) {
        if (w.l2norm)
            row_inv_norms<T>(tk, len, warp, 4, lane, sRK);
        else if (tid < C)
            sRK[tid] = 1.f;
    }
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
        if (lane < len) w.g_cs[(tok0 + lane) * Hv + j] = x0;
        if (lane + 32 < len) w.g_cs[(tok0 + lane + 32) * Hv + j] = x1;
    }
    __syncthreads();
    auto store_norms = [&]() {
        if (w.l2norm && tid < len) {
            if (w.rk_out) w.rk_out[(tok0 + tid) * Hv + j] = sRK[tid];
            if (w.rq_out && want_p) w.rq_out[(tok0 + tid) * Hv + j] = sRQ[tid];
        }
    };
    if (!want_p) store_norms();

    // ---- P = scale (q^ k^T o exp(G_r - G_s)) for s <= r < len and L = strictly-lower(diag(beta) (k^ k^T o
    //      exp(G_r - G_s))) in one pass (warp w owns rows 16w..16w+15, column tiles at or left of the diagonal):
    //      both products take the same K fragments, and each decay factor serves both.  P is staged as rows
    //      in the not yet used A^-1 buffer and stored row by row; L goes over the Q tile once every warp has
    //      read its fragments.
    const bool want_a = w.A_out != nullptr;
    if (want_p) {
        float accp[8][4], accl[8][4];
        zero_acc<8>(accp);
        zero_acc<8>(accl);
        const int r0 = warp * 16;
        // sums of squares of this thread's fragment entries: rows r0 + gq (lo) and r0 + gq + 8 (hi) of q and k
        float sq_lo = 0.f, sq_hi = 0.f, sk_lo = 0.f, sk_hi = 0.f;
        auto ssq = [](uint32_t u) {
            const float2 x = Elt<T>::unpack(u);
            return x.x * x.x + x.y * x.y;
        };
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t aq[4], ak[4];
            load_a(aq, tqt, r0, ks * 16, false, lane);
            load_a(ak, tk, r0, ks * 16, false, lane);
            sq_lo += ssq(aq[0]) + ssq(aq[2]);
            sq_hi += ssq(aq[1]) + ssq(aq[3]);
            sk_lo += ssq(ak[0]) + ssq(ak[2]);
            sk_hi += ssq(ak[1]) + ssq(ak[3]);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                if (np <= warp) {
                    uint32_t b[4];
                    load_b2(b, tk, np * 16, ks * 16, false, lane);
                    mma16816<T>(accp[2 * np], aq, b[0], b[1]);
                    mma16816<T>(accp[2 * np + 1], aq, b[2], b[3]);
                    if (want_a) {
                        mma16816<T>(accl[2 * np], ak, b[0], b[1]);
                        mma16816<T>(accl[2 * np + 1], ak, b[2], b[3]);
                    }
                }
            }
        }
        // the four lanes of a row group (tq) hold disjoint columns of the same two rows
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
            sq_lo += __shfl_xor_sync(0xffffffffu, sq_lo, o);
            sq_hi += __shfl_xor_sync(0xffffffffu, sq_hi, o);
            sk_lo += __shfl_xor_sync(0xffffffffu, sk_lo, o);
            sk_hi += __shfl_xor_sync(0xffffffffu, sk_hi, o);
        }
        if (tq == 0) {
            sRQ[r0 + gq] = w.l2norm ? 1.0f / sqrtf(sq_lo + L2_EPS) : 1.f;
            sRQ[r0 + gq + 8] = w.l2norm ? 1.0f / sqrtf(sq_hi + L2_EPS) : 1.f;
            sRK[r0 + gq] = w.l2norm ? 1.0f / sqrtf(sk_lo + L2_EPS) : 1.f;
            sRK[r0 + gq + 8] = w.l2norm ? 1.0f / sqrtf(sk_hi + L2_EPS) : 1.f;
        }
        __syncthreads();  // every warp has its Q and K fragments (the Q tile may become L) and the norms are in
        store_norms();
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = r0 + gq + 8 * hh, s0 = nt * 8 + tq * 2;
                const float g0 = __expf(sG[r] - sG[s0]), g1 = __expf(sG[r] - sG[s0 + 1]);
                const float rr = w.scale * sRQ[r];
                const float v0 = (s0 <= r && r < len) ? rr * sRK[s0] * g0 * accp[nt][2 * hh] : 0.f;
                const float v1 = (s0 + 1 <= r && r < len) ? rr * sRK[s0 + 1] * g1 * accp[nt][2 * hh + 1] : 0.f;
                *reinterpret_cast<uint32_t *>(sp + r * LDP + s0) = Elt<T>::pack(v0, v1);
                if (want_a) {
                    const float lr = sB[r] * sRK[r];
                    Lm[r * LDF + s0] = (s0 < r && r < len) ? lr * sRK[s0] * g0 * accl[nt][2 * hh] : 0.f;
                    Lm[r * LDF + s0 + 1] = (s0 + 1 < r && r < len) ? lr * sRK[s0 + 1] * g1 * accl[nt][2 * hh + 1] : 0.f;
                }
            }
        __syncthreads();
        for (int i = tid; i < C * 8; i += 128) {
            const int r = i >> 3, c0 = (i & 7) * 8;
            if (r >= len) continue;
            *reinterpret_cast<uint4 *>(static_cast<T *>(w.P_out) + ((tok0 + r) * Hv + j) * C + c0) =
                *reinterpret_cast<const uint4 *>(sp + r * LDP + c0);
        }
        __syncthreads();  // the staging rows are read: the A^-1 buffer is free
    }

    if (want_a) {
        if (!want_p) {
            // ---- L alone (warp w owns rows 16w..16w+15; only column tiles at or left of the diagonal)
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
                        if (s < r && r < len) val = sB[r] * sRK[r] * sRK[s] * __expf(sG[r] - sG[s]) * acc[nt][2 * hh + e];
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
            uint32_t wv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c = c0 + 2 * e;
                const float lo = (c <= r) ? Ai[r * LDF + c] : 0.f;
                const float hi = (c + 1 <= r) ? Ai[r * LDF + c + 1] : 0.f;
                wv[e] = Elt<T>::pack(lo, hi);
            }
            *reinterpret_cast<uint4 *>(static_cast<T *>(w.A_out) + ((tok0 + r) * Hv + j) * C + c0) =
                make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
    }

}

// ============================================================================ launchers

template <typename T>
static cudaError_t wy_fwd_t(const Args &a, const WyArgs &w, cudaStream_t s) {
    if (a.max_chunks == 0) return cudaSuccess;
    auto kern = wy_fwd_kernel<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, WY_SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)a.max_chunks, a.Hv);
    return launch_overlapped(kern, grid, dim3(128), WY_SMEM, s, make_geo(a), w);
}

cudaError_t launch_wy_fwd(const Args &a, const void *q, const void *k, const void *g, const void *beta, float *g_cs,
                          void *A, void *P, float *rq, float *rk, cudaStream_t s) {
    WyArgs w;
    w.q = q;
    w.k = k;
    w.g = g;
    w.beta = beta;
    w.gate_f32 = a.gate_f32;
    w.l2norm = a.l2norm;
    w.scale = a.scale;
    w.g_cs = g_cs;
    w.A_out = A;
    w.P_out = P;
    w.rq_out = rq;
    w.rk_out = rk;
    return a.bf16 ? wy_fwd_t<__nv_bfloat16>(a, w, s) : wy_fwd_t<__half>(a, w, s);
}

}  // namespace gdr
