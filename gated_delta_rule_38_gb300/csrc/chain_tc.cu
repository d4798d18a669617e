// Forward recurrence on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// One CTA of 512 threads per (sequence, value head).  The state is held
// transposed, S = h^T [V x K] in fp32 registers: row e lives in threads e,
// e + 128, e + 256 and e + 384 (a quarter of the key columns each), and row e is
// also TMEM lane e of every [V x *] accumulator.  Per
// chunk of 64 tokens (G = chunk-local cumsum of g, Gl = G at the last valid
// row), with single-thread MMA issue and three MMA rounds:
//
//   round 1:  [Q;K] K^T  -> P = (Q K^T) o Gamma o M (lower, decayed)       (M=128,N=64,K=128)
//             W^T = K^T (A diag(beta e^G))^T                               (M=128,N=64,K=64)
//             U^T = V^T (A diag(beta))^T                                   (M=128,N=64,K=64)
//   round 2:  Delta^T = U^T - S W^T                                        (M=128,N=64,K=128)
//             O1 = S Q^T                                                   (M=128,N=64,K=128)
//   round 3:  X = (Delta^T diag(e^{Gl-G})) K                               (M=128,N=128,K=64)
//             O2 = Delta^T P^T                                             (M=128,N=64,K=64)
//   epilogue: o_r = scale (e^{G_r} O1[:,r] + O2[:,r]);  S <- e^{Gl} S + X
//
// This is the chunk form of S_t = e^{g_t} S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
// o_t = scale S_t q_t, with A = (I + strictly-lower(diag(beta) (K K^T o Gamma)))^-1 from wy_fwd.
#include <cuda_runtime.h>

#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tmap.h"
#include "umma.cuh"

namespace gdr {
namespace {

// ---- shared-memory layout (bytes from a 1024-aligned base)
// stage (x2): [Q b0][K b0][Q b1][K b1] (8 KB each: 64 rows x 128 B), [V b0][V b1], A (64x64), G[64], beta[64]
constexpr uint32_t ST_QK = 0, ST_V = 32768, ST_A = 49152, ST_G = 57344, ST_B = 57600, ST_BYTES = 58368;
constexpr uint32_t P_AKG = 2 * ST_BYTES, P_AB = P_AKG + 8192, P_S = P_AB + 8192, P_W = P_S + 32768,
                   P_P = P_W + 16384, P_D = P_P + 8192, P_DT = P_D + 16384, P_FAC = P_DT + 16384, P_BAR = P_FAC + 512,
                   P_SLOT = P_BAR + 8, P_FLAG = P_SLOT + 4, P_SBAR = P_FLAG + 4, SMEM_USED = P_SBAR + 16;
constexpr int NT = 512;       // threads per CTA: four per TMEM lane
constexpr int QN = NT / 128;  // threads sharing a TMEM lane (state row)
constexpr int SW = DK / QN;   // state columns per thread
constexpr int EW = C / QN;    // columns per thread of a 64-wide accumulator
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for aligning the base

// ---- TMEM columns
constexpr uint32_t T_QK = 0, T_W = 64, T_U = 128, T_O1 = 192, T_O2 = 256, T_X = 320, T_COLS = 512;

struct TcP {
    CUtensorMap tq, tk, tv, ta;  // TMA maps of q, k ([tokens][Hq][K]), v ([tokens][Hv][V]), A ([tokens][Hv][64])
    const void *q, *k, *v, *A, *beta;
    const float *g_cs, *h0;
    void *o, *h;
    void *delta;  // optional [rows,Hv,64,128]: Delta = U - W h of every chunk
    float *fin;
    // sequence split into nseg segments of whole chunks (1 = no split):
    //   affine pass: block x = 2*seg + kind; kind 0 starts from zero, kind 1 from the identity with
    //                zero values; both write their end state (S-form [V][K] fp32) to seg_end[kind]
    //   full pass  : block x = seg; starts from seg_start (S-form) when given
    int nseg;
    const float *seg_start;  // [N,Hv,nseg,128,128]
    float *seg_end0, *seg_end1;
    bool gate_f32, l2norm, v_first, h_api;
    float scale;
};

// Copy `valid` rows of a [64 x 128] bf16/fp16 row block (row stride in elements)
// into two swizzled 64-column blocks that are `bstride` bytes apart; rows past
// `valid` are zero-filled.
template <typename T>
__device__ __forceinline__ void load_tile128(uint32_t dst, uint32_t bstride, const T *src, long long stride, int valid,
                                             int tid) {
#pragma unroll
    for (int i = tid; i < 64 * 16; i += NT) {
        const int r = i >> 4, c = i & 15;
        const bool ok = r < valid;
        cp_async16(dst + (uint32_t)(c >> 3) * bstride + umma::off(r, (c & 7) * 8, 0), ok ? src + r * stride + c * 8 : src,
                   ok);
    }
}
template <typename T>
__device__ __forceinline__ void load_tile64(uint32_t dst, const T *src, long long stride, int valid, int tid) {
#pragma unroll
    for (int i = tid; i < 64 * 8; i += NT) {
        const int r = i >> 3, c = i & 7;
        const bool ok = r < valid;
        cp_async16(dst + umma::off(r, c * 8, 0), ok ? src + r * stride + c * 8 : src, ok);
    }
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, bool valid) {
    const int n = valid ? 4 : 0;
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}

// In-place x / sqrt(sum x^2 + eps) of `rows` rows of a [64 x 128] swizzled tile
// (two 64-column blocks `bstride` apart).  Lane l of a warp takes a quarter
// (32 values) of row 8*pass + l/4.
template <typename T>
__device__ __forceinline__ void l2norm_tile(uint32_t base, uint32_t bstride, int rows, int warp, int lane) {
    const int rq = lane >> 2, qq = lane & 3;
    for (int r0 = warp * 8; r0 < rows; r0 += 8 * (NT / 32)) {
        const int r = r0 + rq;
        uint32_t addr[4];
        uint4 u[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int ch = qq * 4 + c;  // 16-byte chunk 0..15 of the row
            addr[c] = base + (uint32_t)(ch >> 3) * bstride + umma::off(r, (ch & 7) * 8, 0);
            u[c] = umma::ld_shared_v4(addr[c]);
        }
        float ss = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t w[4] = {u[c].x, u[c].y, u[c].z, u[c].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 x = Elt<T>::unpack(w[e]);
                ss += x.x * x.x + x.y * x.y;
            }
        }
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        const float inv = 1.0f / sqrtf(ss + L2_EPS);
        if (r < rows) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t w[4] = {u[c].x, u[c].y, u[c].z, u[c].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 x = Elt<T>::unpack(w[e]);
                    w[e] = Elt<T>::pack(x.x * inv, x.y * inv);
                }
                umma::st_shared_v4(addr[c], w[0], w[1], w[2], w[3]);
            }
        }
    }
}

// Write 16 fp32 values as columns col0..col0+15 (col0 a multiple of 16) of a swizzled row.
template <typename T>
__device__ __forceinline__ void store16(uint32_t base, int row, int col0, const float *x) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        umma::st_shared_v4(base + umma::off(row, col0 + c * 8, 0), Elt<T>::pack(x[c * 8], x[c * 8 + 1]),
                           Elt<T>::pack(x[c * 8 + 2], x[c * 8 + 3]), Elt<T>::pack(x[c * 8 + 4], x[c * 8 + 5]),
                           Elt<T>::pack(x[c * 8 + 6], x[c * 8 + 7]));
    }
}

template <typename T> struct IsBf16 { static constexpr bool value = false; };
template <> struct IsBf16<__nv_bfloat16> { static constexpr bool value = true; };

__device__ __forceinline__ void sync_tc() {
    umma::fence_async_smem();
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
}

template <typename T, bool WRITE_O, bool AFFINE>
__device__ __forceinline__ void chain_fwd_body(const Geo &geo, const TcP &p, const int bx, const int j, const int n) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const int Hv = geo.Hv, Hq = geo.Hq, hq = j / (Hv / Hq);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // thread (e, qq): TMEM lane / state row e, column quarter qq
    const int e = tid & 127, qq = tid >> 7, lb = (warp & 3) * 32;
    constexpr bool bf16 = IsBf16<T>::value;
    long long tok0;
    int len, row0;
    geo.seq(n, tok0, len, row0);
    const int nc_all = (len + C - 1) / C;
    // this block's segment of chunks [cb, ce)
    const int seg = AFFINE ? bx >> 1 : bx;
    const int kind = AFFINE ? bx & 1 : 0;  // 1: identity start, zero values
    const int sl = (nc_all + p.nseg - 1) / p.nseg;
    const int cb = min(nc_all, seg * sl), ce = min(nc_all, cb + sl);
    const long long st_base = ((long long)n * Hv + j) * DK * DV;
    const long long seg_base = (((long long)n * Hv + j) * p.nseg + seg) * DK * DV;
    const uint32_t bar = sb + P_BAR;
    volatile int *sflag = reinterpret_cast<volatile int *>(smem + P_FLAG);
    float *fEG = reinterpret_cast<float *>(smem + P_FAC);  // e^{G_s}
    float *fEL = fEG + C;                                   // e^{Gl - G_s}

    const bool use_v = !(AFFINE && kind == 1);  // the identity-start affine pass has zero values
    if (tid == 0) {
        umma::mbar_init(bar, 1);
        umma::mbar_init(sb + P_SBAR, 1);
        umma::mbar_init(sb + P_SBAR + 8, 1);
        umma::fence_mbar_init();
        *sflag = 0;
    }
    if (warp == 0) umma::alloc(sb + P_SLOT, T_COLS);
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + P_SLOT);

    // fp32 state: S[e][SW*qq + i] = h[SW*qq + i][e]
    float S[SW];
#pragma unroll
    for (int i = 0; i < SW; ++i) {
        const int d = qq * SW + i;
        if (AFFINE)
            S[i] = (kind == 1 && d == e) ? 1.f : 0.f;
        else if (p.seg_start)
            S[i] = p.seg_start[seg_base + (long long)e * DK + d];
        else
            S[i] = p.h0 ? p.h0[st_base + (p.v_first ? (long long)e * DK + d : (long long)d * DV + e)] : 0.f;
    }
    auto write_S_tile = [&]() {
#pragma unroll
        for (int c = 0; c < SW; c += 16) {
            const int col = qq * SW + c;
            store16<T>(sb + P_S + (col >> 6) * 16384, e, col & 63, S + c);
        }
    };
    write_S_tile();

    float breg = 0.f;
    uint32_t sphase[2] = {0u, 0u};
    unsigned pend = 0;  // stages with a tile load in flight
    auto prefetch = [&](int i) {
        const uint32_t st = sb + (i & 1) * ST_BYTES, sbar = sb + P_SBAR + (i & 1) * 8;
        pend |= 1u << (i & 1);
        const long long tb = tok0 + (long long)i * C;
        const int valid = min(C, len - i * C);
        if (tid == 0) {
            // tiles of 64 rows x 128 bytes land in the 128-byte-swizzled layout the MMAs read
            tma::expect_tx(sbar, (WRITE_O ? 16384u : 0u) + 16384u + (use_v ? 16384u : 0u) + 8192u);
            const int t = (int)tb;
            if (WRITE_O) {
                tma::load3d(st + ST_QK, &p.tq, 0, hq, t, sbar);
                tma::load3d(st + ST_QK + 16384, &p.tq, 64, hq, t, sbar);
            }
            tma::load3d(st + ST_QK + 8192, &p.tk, 0, hq, t, sbar);
            tma::load3d(st + ST_QK + 24576, &p.tk, 64, hq, t, sbar);
            if (use_v) {
                tma::load3d(st + ST_V, &p.tv, 0, j, t, sbar);
                tma::load3d(st + ST_V + 8192, &p.tv, 64, j, t, sbar);
            }
            tma::load3d(st + ST_A, &p.ta, 0, j, t, sbar);
        }
        if (tid < C) {
            const bool ok = tid < valid;
            cp_async4(st + ST_G + tid * 4, p.g_cs + (ok ? (tb + tid) * Hv + j : 0), ok);
            breg = ok ? load_gate<T>(p.beta, (tb + tid) * Hv + j, p.gate_f32) : 0.f;
        }
        cp_async_commit();
    };
    if (cb < ce) prefetch(cb);

    uint32_t phase = 0;
    const uint32_t id_n64 = umma::idesc(128, 64, bf16, false, false);
    const uint32_t id_n64_amn = umma::idesc(128, 64, bf16, true, false);
    const uint32_t id_n64_bmn = umma::idesc(128, 64, bf16, false, true);
    const uint32_t id_n128_bmn = umma::idesc(128, 128, bf16, false, true);
    // descriptors of the persistent operand tiles
    const uint64_t dAKG = umma::desc(sb + P_AKG, 16, 1024), dAB = umma::desc(sb + P_AB, 16, 1024);
    const uint64_t dS = umma::desc(sb + P_S, 16, 1024), dW = umma::desc(sb + P_W, 8192, 1024);
    const uint64_t dD = umma::desc(sb + P_D, 16, 1024), dDT = umma::desc(sb + P_DT, 16, 1024);
    const uint64_t dP = umma::desc(sb + P_P, 16, 1024);
    // one thread waits for the MMAs; the block then meets at a barrier
    auto wait_mma = [&]() -> bool {
        if (tid == 0 && !umma::mbar_wait(bar, phase)) {
            raise_error(geo.err, GDR_ERR_TIMEOUT);
            *sflag = 1;
        }
        phase ^= 1;
        umma::fence_before();
        __syncthreads();
        umma::fence_after();
        return *sflag == 0;
    };

    for (int i = cb; i < ce; ++i) {
        const uint32_t st = sb + (i & 1) * ST_BYTES;
        const float *sG = reinterpret_cast<const float *>(smem + (i & 1) * ST_BYTES + ST_G);
        float *sB = reinterpret_cast<float *>(smem + (i & 1) * ST_BYTES + ST_B);
        cp_async_wait<0>();
        if (tid < C) sB[tid] = breg;
        if (!umma::mbar_wait(sb + P_SBAR + (i & 1) * 8, sphase[i & 1])) {
            raise_error(geo.err, GDR_ERR_TIMEOUT);
            *sflag = 1;
        }
        sphase[i & 1] ^= 1u;
        pend &= ~(1u << (i & 1));
        __syncthreads();
        if (*sflag) break;
        const int valid = min(C, len - i * C);
        const float Gl = sG[valid - 1];
        if (p.l2norm) {
            if (WRITE_O) l2norm_tile<T>(st + ST_QK, 16384, valid, warp, lane);
            l2norm_tile<T>(st + ST_QK + 8192, 16384, valid, warp, lane);
        }
        if (tid < C) {
            fEG[tid] = __expf(sG[tid]);
            fEL[tid] = __expf(Gl - sG[tid]);
        }
        // scaled copies of A: columns s times beta_s e^{G_s} (for W) and beta_s (for U)
#pragma unroll
        for (int u = 0; u < (C * 8) / NT; ++u) {
            const int ci = tid + u * NT, r = ci >> 3, c = ci & 7;
            const uint32_t o = umma::off(r, c * 8, 0);
            uint4 a = umma::ld_shared_v4(st + ST_A + o);
            if (r >= valid) a = make_uint4(0u, 0u, 0u, 0u);
            const uint32_t w[4] = {a.x, a.y, a.z, a.w};
            uint32_t wk[4], wb[4];
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2) {
                const int s = c * 8 + 2 * q2;
                const float2 x = Elt<T>::unpack(w[q2]);
                const float b0 = sB[s], b1 = sB[s + 1];
                wb[q2] = Elt<T>::pack(x.x * b0, x.y * b1);
                wk[q2] = Elt<T>::pack(x.x * b0 * __expf(sG[s]), x.y * b1 * __expf(sG[s + 1]));
            }
            umma::st_shared_v4(sb + P_AKG + o, wk[0], wk[1], wk[2], wk[3]);
            umma::st_shared_v4(sb + P_AB + o, wb[0], wb[1], wb[2], wb[3]);
        }
        // the state before this chunk (optional output)
        if (!AFFINE && p.h) {
            T *h = static_cast<T *>(p.h);
            const long long hb = ((long long)(row0 + i) * Hv + j) * DK * DV;
            if (p.h_api && p.v_first) {
                T *hr = h + hb + (long long)e * DK + qq * SW;
#pragma unroll
                for (int d = 0; d < SW; d += 8) {
                    uint4 w;
                    w.x = Elt<T>::pack(S[d], S[d + 1]);
                    w.y = Elt<T>::pack(S[d + 2], S[d + 3]);
                    w.z = Elt<T>::pack(S[d + 4], S[d + 5]);
                    w.w = Elt<T>::pack(S[d + 6], S[d + 7]);
                    *reinterpret_cast<uint4 *>(hr + d) = w;
                }
            } else {
                T *hc = h + hb + (long long)(qq * SW) * DV + e;
#pragma unroll
                for (int d = 0; d < SW; ++d) hc[d * DV] = Elt<T>::from_f(S[d]);
            }
        }
        sync_tc();
        if (i + 1 < ce) prefetch(i + 1);

        // ---- round 1
        // (descriptors of successive K-steps differ only in the start-address field: add offset >> 4)
        const uint64_t dQa = umma::desc(st + ST_QK, 16, 1024), dKa = umma::desc(st + ST_QK + 8192, 16, 1024);
        const uint64_t dKmn = umma::desc(st + ST_QK + 8192, 16384, 1024), dVmn = umma::desc(st + ST_V, 8192, 1024);
        if (tid == 0) {
            if (WRITE_O) {
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t ko = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
                    umma::mma(tmem + T_QK, dQa + ko, dKa + ko, id_n64, ks > 0);
                }
            }
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                umma::mma(tmem + T_W, dKmn + ks * 128, dAKG + ks * 2, id_n64_amn, ks > 0);
                if (use_v) umma::mma(tmem + T_U, dVmn + ks * 128, dAB + ks * 2, id_n64_amn, ks > 0);
            }
            umma::commit(bar);
        }
        if (!wait_mma()) break;
#pragma unroll
        for (int c = 0; c < EW; c += 16) {
            // -W row d = e, token columns EW*qq + c .. : MN-major operand rows (key index d)
            float x[16];
            umma::ld16(umma::taddr(tmem, lb, T_W + qq * EW + c), x);
            umma::ld_wait();
#pragma unroll
            for (int u = 0; u < 16; ++u) x[u] = -x[u];
            store16<T>(sb + P_W, e, qq * EW + c, x);
        }
        if (WRITE_O && e < C) {
            const int r = e;
            const float gr = sG[r];
#pragma unroll
            for (int c = 0; c < EW; c += 16) {
                float x[16];
                umma::ld16(umma::taddr(tmem, lb, T_QK + qq * EW + c), x);
                umma::ld_wait();
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int s = qq * EW + c + u;
                    x[u] = (s <= r && r < valid) ? x[u] * __expf(gr - sG[s]) : 0.f;
                }
                store16<T>(sb + P_P, r, qq * EW + c, x);
            }
        }
        sync_tc();

        // ---- round 2: Delta^T = U^T + S (-W)^T ;  O1 = S Q^T
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t so = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
                umma::mma(tmem + T_U, dS + so, dW + ks * 128, id_n64_bmn, use_v || ks > 0);
                if (WRITE_O) umma::mma(tmem + T_O1, dS + so, dQa + so, id_n64, ks > 0);
            }
            umma::commit(bar);
        }
        if (!wait_mma()) break;
#pragma unroll
        for (int c = 0; c < EW; c += 16) {
            float x[16], y[16];
            umma::ld16(umma::taddr(tmem, lb, T_U + qq * EW + c), x);
            umma::ld_wait();
#pragma unroll
            for (int u = 0; u < 16; ++u) y[u] = x[u] * fEL[qq * EW + c + u];
            store16<T>(sb + P_D, e, qq * EW + c, x);
            store16<T>(sb + P_DT, e, qq * EW + c, y);
            if (!AFFINE && p.delta) {
                T *dr = static_cast<T *>(p.delta) + ((long long)(row0 + i) * Hv + j) * C * DV +
                        (long long)(qq * EW + c) * DV + e;
#pragma unroll
                for (int u = 0; u < 16; ++u) dr[u * DV] = Elt<T>::from_f(x[u]);
            }
        }
        sync_tc();

        // ---- round 3: X = Delta~^T K ;  O2 = Delta^T P^T
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                umma::mma(tmem + T_X, dDT + ks * 2, dKmn + ks * 128, id_n128_bmn, ks > 0);
                if (WRITE_O) umma::mma(tmem + T_O2, dD + ks * 2, dP + ks * 2, id_n64, ks > 0);
            }
            umma::commit(bar);
        }
        if (!wait_mma()) break;
        {
            const float eg = __expf(Gl);
#pragma unroll
            for (int c = 0; c < SW; c += 16) {
                float x[16];
                umma::ld16(umma::taddr(tmem, lb, T_X + qq * SW + c), x);
                umma::ld_wait();
#pragma unroll
                for (int u = 0; u < 16; ++u) S[c + u] = eg * S[c + u] + x[u];
            }
            if (WRITE_O) {
                T *o = static_cast<T *>(p.o) + ((tok0 + (long long)i * C + qq * EW) * Hv + j) * geo.V + e;
                const long long ostride = (long long)Hv * geo.V;
#pragma unroll
                for (int c = 0; c < EW; c += 16) {
                    float x1[16], x2[16];
                    umma::ld16(umma::taddr(tmem, lb, T_O1 + qq * EW + c), x1);
                    umma::ld16(umma::taddr(tmem, lb, T_O2 + qq * EW + c), x2);
                    umma::ld_wait();
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const int r = qq * EW + c + u;
                        if (r < valid && e < geo.V)
                            o[(c + u) * ostride] = Elt<T>::from_f(p.scale * (fEG[r] * x1[u] + x2[u]));
                    }
                }
            }
            write_S_tile();
        }
        sync_tc();
    }

    if (*sflag == 0) {
        if (AFFINE) {
            float *dst = (kind ? p.seg_end1 : p.seg_end0) + seg_base + (long long)e * DK + qq * SW;
#pragma unroll
            for (int i = 0; i < SW; i += 4) *reinterpret_cast<float4 *>(dst + i) = make_float4(S[i], S[i + 1], S[i + 2], S[i + 3]);
        } else if (p.fin && seg == p.nseg - 1) {
#pragma unroll
            for (int i = 0; i < SW; ++i) {
                const int d = qq * SW + i;
                p.fin[st_base + (p.v_first ? (long long)e * DK + d : (long long)d * DV + e)] = S[i];
            }
        }
    }
    // after an error, let tile loads still in flight land before the block exits (bounded)
    for (int st2 = 0; st2 < 2; ++st2)
        if (pend & (1u << st2)) umma::mbar_wait(sb + P_SBAR + st2 * 8, sphase[st2], 4000000L);
    umma::fence_before();
    __syncthreads();
    if (warp == 0) umma::dealloc(tmem, T_COLS);
}

// ============================================================================ reverse chain
//
// One CTA of 512 threads per (sequence, value head); chunks in reverse order;
// dS = dH^T [V x K] (gradient w.r.t. the transposed state) in fp32 registers,
// thread (e, qq) holding row e, key quarter qq.  With dS' the gradient arriving at
// the end of the chunk, K~ = diag(e^{Gl-G}) K and P = (Q K^T) o Gamma o M:
//
//   round 1:  [K;Q] Q^T -> P^T rows (scaled, upper part)                  (M=128,N=64,K=128)
//             W^T = K^T (A diag(beta e^G))^T                              (M=128,N=64,K=64)
//             E1 = dS' K^T                                                (M=128,N=64,K=128)
//   round 2:  E2 = dO^T P                                                 (M=128,N=64,K=64)
//             dDelta^T = E1 diag(e^{Gl-G}) + E2
//   round 3:  X = (scale dO diag(e^G))^T Q - dDelta^T W                   (M=128,N=128,K=64 x2)
//   epilogue: dS <- e^{Gl} dS' + X
// It stores dS' of every chunk (the gradient w.r.t. the state after the chunk)
// for the per-chunk gradient kernel; the last dS is dh0.

struct TcBwdP {
    CUtensorMap tq, tk, tdo, ta;  // TMA maps of q, k, dO, A
    const void *q, *k, *A, *beta, *dout;
    const float *g_cs, *dht;
    void *dhn;
    void *ddelta;  // [rows,Hv,64,128]: dDelta of every chunk
    float *dh0;
    bool gate_f32, l2norm, v_first;
    float scale;
    // sequence split, mirrored: segment seg covers chunks [cb, ce), walked from ce-1 down to cb;
    // the affine pass (block x = 2*seg + kind; kind 1 = identity start with dO = 0) writes the
    // gradient at the segment start; the full pass starts from seg_start at the segment end
    int nseg;
    const float *seg_start;
    float *seg_end0, *seg_end1;
};

// persistent tiles of the reverse chain (same stage layout as the forward, with
// [K b][Q b] order in the 32 KB block and dO in place of V)
constexpr uint32_t B_AKG = 2 * ST_BYTES, B_DS = B_AKG + 8192, B_WT = B_DS + 32768, B_PT = B_WT + 16384,
                   B_DOG = B_PT + 8192, B_DDT = B_DOG + 16384, B_FAC = B_DDT + 16384, B_BAR = B_FAC + 512,
                   B_SLOT = B_BAR + 8, B_FLAG = B_SLOT + 4, B_SBAR = B_FLAG + 4, B_USED = B_SBAR + 16;
constexpr uint32_t B_SMEM_BYTES = B_USED + 1024;
constexpr uint32_t TB_KQ = 0, TB_W = 64, TB_E1 = 128, TB_E2 = 192, TB_X = 256, TB_COLS = 512;

template <typename T, bool AFFINE>
__device__ __forceinline__ void chain_bwd_body(const Geo &geo, const TcBwdP &p, const int bx, const int j, const int n) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const int Hv = geo.Hv, Hq = geo.Hq, hq = j / (Hv / Hq);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int e = tid & 127, qq = tid >> 7, lb = (warp & 3) * 32;
    constexpr bool bf16 = IsBf16<T>::value;
    long long tok0;
    int len, row0;
    geo.seq(n, tok0, len, row0);
    const int nc_all = (len + C - 1) / C;
    const int seg = AFFINE ? bx >> 1 : bx;
    const int kind = AFFINE ? bx & 1 : 0;
    const int sl = (nc_all + p.nseg - 1) / p.nseg;
    const int cb = min(nc_all, seg * sl), ce = min(nc_all, cb + sl);
    const long long st_base = ((long long)n * Hv + j) * DK * DV;
    const long long seg_base = (((long long)n * Hv + j) * p.nseg + seg) * DK * DV;
    const uint32_t bar = sb + B_BAR;
    volatile int *sflag = reinterpret_cast<volatile int *>(smem + B_FLAG);
    float *fEG = reinterpret_cast<float *>(smem + B_FAC);
    float *fEL = fEG + C;

    const bool use_do = !(AFFINE && kind == 1);  // the identity-start affine pass has dO = 0
    if (tid == 0) {
        umma::mbar_init(bar, 1);
        umma::mbar_init(sb + B_SBAR, 1);
        umma::mbar_init(sb + B_SBAR + 8, 1);
        umma::fence_mbar_init();
        *sflag = 0;
    }
    if (warp == 0) umma::alloc(sb + B_SLOT, TB_COLS);
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + B_SLOT);

    float S[SW];  // dS[e][SW*qq + i] = dH[SW*qq + i][e]
#pragma unroll
    for (int i = 0; i < SW; ++i) {
        const int d = qq * SW + i;
        if (AFFINE)
            S[i] = (kind == 1 && d == e) ? 1.f : 0.f;
        else if (p.seg_start)
            S[i] = p.seg_start[seg_base + (long long)e * DK + d];
        else
            S[i] = p.dht ? p.dht[st_base + (p.v_first ? (long long)e * DK + d : (long long)d * DV + e)] : 0.f;
    }
    auto write_S_tile = [&]() {
#pragma unroll
        for (int c = 0; c < SW; c += 16) {
            const int col = qq * SW + c;
            store16<T>(sb + B_DS + (col >> 6) * 16384, e, col & 63, S + c);
        }
    };
    write_S_tile();

    float breg = 0.f;
    uint32_t sphase[2] = {0u, 0u};
    unsigned pend = 0;  // stages with a tile load in flight
    auto prefetch = [&](int i) {
        const uint32_t st = sb + (i & 1) * ST_BYTES, sbar = sb + B_SBAR + (i & 1) * 8;
        pend |= 1u << (i & 1);
        const long long tb = tok0 + (long long)i * C;
        const int valid = min(C, len - i * C);
        if (tid == 0) {
            tma::expect_tx(sbar, 16384u + 16384u + (use_do ? 16384u : 0u) + 8192u);
            const int t = (int)tb;
            tma::load3d(st + ST_QK, &p.tk, 0, hq, t, sbar);
            tma::load3d(st + ST_QK + 16384, &p.tk, 64, hq, t, sbar);
            tma::load3d(st + ST_QK + 8192, &p.tq, 0, hq, t, sbar);
            tma::load3d(st + ST_QK + 24576, &p.tq, 64, hq, t, sbar);
            if (use_do) {
                tma::load3d(st + ST_V, &p.tdo, 0, j, t, sbar);
                tma::load3d(st + ST_V + 8192, &p.tdo, 64, j, t, sbar);
            }
            tma::load3d(st + ST_A, &p.ta, 0, j, t, sbar);
        }
        if (tid < C) {
            const bool ok = tid < valid;
            cp_async4(st + ST_G + tid * 4, p.g_cs + (ok ? (tb + tid) * Hv + j : 0), ok);
            breg = ok ? load_gate<T>(p.beta, (tb + tid) * Hv + j, p.gate_f32) : 0.f;
        }
        cp_async_commit();
    };
    if (cb < ce) prefetch(ce - 1);

    uint32_t phase = 0;
    const uint32_t id_n64 = umma::idesc(128, 64, bf16, false, false);
    const uint32_t id_n64_amn = umma::idesc(128, 64, bf16, true, false);
    const uint32_t id_n128_ab_mn = umma::idesc(128, 128, bf16, true, true);
    const uint32_t id_n128 = umma::idesc(128, 128, bf16, false, false);
    const uint64_t dAKG = umma::desc(sb + B_AKG, 16, 1024), dDS = umma::desc(sb + B_DS, 16, 1024);
    const uint64_t dWT = umma::desc(sb + B_WT, 16, 1024), dPT = umma::desc(sb + B_PT, 16, 1024);
    const uint64_t dOG = umma::desc(sb + B_DOG, 8192, 1024), dDDT = umma::desc(sb + B_DDT, 16, 1024);
    auto wait_mma = [&]() -> bool {
        if (tid == 0 && !umma::mbar_wait(bar, phase)) {
            raise_error(geo.err, GDR_ERR_TIMEOUT);
            *sflag = 1;
        }
        phase ^= 1;
        umma::fence_before();
        __syncthreads();
        umma::fence_after();
        return *sflag == 0;
    };

    for (int i = ce - 1; i >= cb; --i) {
        const uint32_t st = sb + (i & 1) * ST_BYTES;
        const float *sG = reinterpret_cast<const float *>(smem + (i & 1) * ST_BYTES + ST_G);
        float *sB = reinterpret_cast<float *>(smem + (i & 1) * ST_BYTES + ST_B);
        cp_async_wait<0>();
        if (tid < C) sB[tid] = breg;
        if (!umma::mbar_wait(sb + B_SBAR + (i & 1) * 8, sphase[i & 1])) {
            raise_error(geo.err, GDR_ERR_TIMEOUT);
            *sflag = 1;
        }
        sphase[i & 1] ^= 1u;
        pend &= ~(1u << (i & 1));
        // gradient w.r.t. the state after this chunk, for the per-chunk kernel ([K][V] layout)
        if (!AFFINE) {
            T *hc = static_cast<T *>(p.dhn) + ((long long)(row0 + i) * Hv + j) * DK * DV + (long long)(qq * SW) * DV + e;
#pragma unroll
            for (int d = 0; d < SW; ++d) hc[d * DV] = Elt<T>::from_f(S[d]);
        }
        __syncthreads();
        if (*sflag) break;
        const int valid = min(C, len - i * C);
        const float Gl = sG[valid - 1];
        if (p.l2norm) {
            l2norm_tile<T>(st + ST_QK, 16384, valid, warp, lane);
            l2norm_tile<T>(st + ST_QK + 8192, 16384, valid, warp, lane);
        }
        if (tid < C) {
            fEG[tid] = __expf(sG[tid]);
            fEL[tid] = __expf(Gl - sG[tid]);
        }
#pragma unroll
        for (int u = 0; u < (C * 8) / NT; ++u) {
            const int ci = tid + u * NT, r = ci >> 3, c = ci & 7;
            const uint32_t o = umma::off(r, c * 8, 0);
            uint4 a = umma::ld_shared_v4(st + ST_A + o);
            if (r >= valid) a = make_uint4(0u, 0u, 0u, 0u);
            const uint32_t w[4] = {a.x, a.y, a.z, a.w};
            uint32_t wk[4];
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2) {
                const int s = c * 8 + 2 * q2;
                const float2 x = Elt<T>::unpack(w[q2]);
                wk[q2] = Elt<T>::pack(x.x * sB[s] * __expf(sG[s]), x.y * sB[s + 1] * __expf(sG[s + 1]));
            }
            umma::st_shared_v4(sb + B_AKG + o, wk[0], wk[1], wk[2], wk[3]);
        }
        // scale e^{G_s} dO rows -> dOg (same two-block layout)
#pragma unroll
        for (int u = 0; u < (C * 16) / NT; ++u) {
            const int ci = tid + u * NT, r = ci >> 4, c = ci & 15;
            const uint32_t o = (uint32_t)(c >> 3) * 8192 + umma::off(r, (c & 7) * 8, 0);
            const uint4 a = umma::ld_shared_v4(st + ST_V + o);
            const float f = (r < valid && use_do) ? p.scale * __expf(sG[r]) : 0.f;
            const uint32_t w[4] = {a.x, a.y, a.z, a.w};
            uint32_t wo[4];
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2) {
                const float2 x = Elt<T>::unpack(w[q2]);
                wo[q2] = Elt<T>::pack(x.x * f, x.y * f);
            }
            umma::st_shared_v4(sb + B_DOG + o, wo[0], wo[1], wo[2], wo[3]);
        }
        sync_tc();
        if (i > cb) prefetch(i - 1);

        // ---- round 1: [K;Q] Q^T, W^T, E1 = dS' K^T
        const uint64_t dKa = umma::desc(st + ST_QK, 16, 1024), dQa = umma::desc(st + ST_QK + 8192, 16, 1024);
        const uint64_t dKmn = umma::desc(st + ST_QK, 16384, 1024), dQmn = umma::desc(st + ST_QK + 8192, 16384, 1024);
        const uint64_t dOmn = umma::desc(st + ST_V, 8192, 1024);
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t ko = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
                umma::mma(tmem + TB_KQ, dKa + ko, dQa + ko, id_n64, ks > 0);
                umma::mma(tmem + TB_E1, dDS + ko, dKa + ko, id_n64, ks > 0);
            }
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) umma::mma(tmem + TB_W, dKmn + ks * 128, dAKG + ks * 2, id_n64_amn, ks > 0);
            umma::commit(bar);
        }
        if (!wait_mma()) break;
#pragma unroll
        for (int c = 0; c < EW; c += 16) {
            float x[16];
            umma::ld16(umma::taddr(tmem, lb, TB_W + qq * EW + c), x);
            umma::ld_wait();
            store16<T>(sb + B_WT, e, qq * EW + c, x);
        }
        if (e < C) {
            const int r = e;
            const float gr = sG[r];
#pragma unroll
            for (int c = 0; c < EW; c += 16) {
                float x[16];
                umma::ld16(umma::taddr(tmem, lb, TB_KQ + qq * EW + c), x);
                umma::ld_wait();
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int s2 = qq * EW + c + u;
                    x[u] = (s2 >= r && s2 < valid) ? x[u] * p.scale * __expf(sG[s2] - gr) : 0.f;
                }
                store16<T>(sb + B_PT, r, qq * EW + c, x);
            }
        }
        sync_tc();

        // ---- round 2: E2 = dO^T P
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                if (use_do) umma::mma(tmem + TB_E2, dOmn + ks * 128, dPT + ks * 2, id_n64_amn, ks > 0);
            umma::commit(bar);
        }
        if (!wait_mma()) break;
#pragma unroll
        for (int c = 0; c < EW; c += 16) {
            float x1[16], x2[16];
            umma::ld16(umma::taddr(tmem, lb, TB_E1 + qq * EW + c), x1);
            umma::ld16(umma::taddr(tmem, lb, TB_E2 + qq * EW + c), x2);
            umma::ld_wait();
            if (!use_do) {
#pragma unroll
                for (int u = 0; u < 16; ++u) x2[u] = 0.f;
            }
#pragma unroll
            for (int u = 0; u < 16; ++u) x1[u] = -(x1[u] * fEL[qq * EW + c + u] + x2[u]);
            store16<T>(sb + B_DDT, e, qq * EW + c, x1);
            if (!AFFINE) {
                T *dr = static_cast<T *>(p.ddelta) + ((long long)(row0 + i) * Hv + j) * C * DV +
                        (long long)(qq * EW + c) * DV + e;
#pragma unroll
                for (int u = 0; u < 16; ++u) dr[u * DV] = Elt<T>::from_f(qq * EW + c + u < valid ? -x1[u] : 0.f);
            }
        }
        sync_tc();

        // ---- round 3: X = dOg^T Q - dDelta^T W
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                if (use_do) umma::mma(tmem + TB_X, dOG + ks * 128, dQmn + ks * 128, id_n128_ab_mn, ks > 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) umma::mma(tmem + TB_X, dDDT + ks * 2, dWT + ks * 2, id_n128, use_do || ks > 0);
            umma::commit(bar);
        }
        if (!wait_mma()) break;
        {
            const float eg = __expf(Gl);
#pragma unroll
            for (int c = 0; c < SW; c += 16) {
                float x[16];
                umma::ld16(umma::taddr(tmem, lb, TB_X + qq * SW + c), x);
                umma::ld_wait();
#pragma unroll
                for (int u = 0; u < 16; ++u) S[c + u] = eg * S[c + u] + x[u];
            }
            write_S_tile();
        }
        sync_tc();
    }

    if (*sflag == 0) {
        if (AFFINE) {
            float *dst = (kind ? p.seg_end1 : p.seg_end0) + seg_base + (long long)e * DK + qq * SW;
#pragma unroll
            for (int i = 0; i < SW; i += 4) *reinterpret_cast<float4 *>(dst + i) = make_float4(S[i], S[i + 1], S[i + 2], S[i + 3]);
        } else if (p.dh0 && seg == 0) {
#pragma unroll
            for (int i = 0; i < SW; ++i) {
                const int d = qq * SW + i;
                p.dh0[st_base + (p.v_first ? (long long)e * DK + d : (long long)d * DV + e)] = S[i];
            }
        }
    }
    for (int st2 = 0; st2 < 2; ++st2)
        if (pend & (1u << st2)) umma::mbar_wait(sb + B_SBAR + st2 * 8, sphase[st2], 4000000L);
    umma::fence_before();
    __syncthreads();
    if (warp == 0) umma::dealloc(tmem, TB_COLS);
}

template <typename T, bool WRITE_O, bool AFFINE>
__global__ void __launch_bounds__(NT, 1) chain_fwd_tc_kernel(Geo geo, const __grid_constant__ TcP p) {
    chain_fwd_body<T, WRITE_O, AFFINE>(geo, p, blockIdx.x, blockIdx.y, blockIdx.z);
}

template <typename T, bool AFFINE>
__global__ void __launch_bounds__(NT, 1) chain_bwd_tc_kernel(Geo geo, const __grid_constant__ TcBwdP p) {
    chain_bwd_body<T, AFFINE>(geo, p, blockIdx.x, blockIdx.y, blockIdx.z);
}

template <typename T>
cudaError_t chain_bwd_tc_t(const Args &a, const TcBwdP &p, bool affine, cudaStream_t s) {
    auto kern = affine ? chain_bwd_tc_kernel<T, true> : chain_bwd_tc_kernel<T, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, B_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid(affine ? 2 * p.nseg : p.nseg, a.Hv, a.N);
    return launch_plain(kern, grid, dim3(NT), B_SMEM_BYTES, s, make_geo(a), p);
}

template <typename T>
cudaError_t chain_fwd_tc_t(const Args &a, const TcP &p, bool write_o, bool affine, cudaStream_t s) {
    auto kern = affine ? chain_fwd_tc_kernel<T, false, true>
                       : (write_o ? chain_fwd_tc_kernel<T, true, false> : chain_fwd_tc_kernel<T, false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid(affine ? 2 * p.nseg : p.nseg, a.Hv, a.N);
    return launch_plain(kern, grid, dim3(NT), SMEM_BYTES, s, make_geo(a), p);
}

// Segment start states: S_0 = init (API state layout, or zero), S_{s+1} = S_s P_s + Q_s in fp32,
// walking segments forward (or backward when reverse), with P = seg_end1, Q = seg_end0 (S-form).
// One block of four warps per (16-row slice of the value index, head, sequence); warp w owns rows 4w..4w+3,
// lane l the columns 4l..4l+3, so each row of P_s is read from shared memory once per warp, conflict-free,
// and feeds 16 products per thread.  The walk is serial over the segments, so each segment's P_s (64 KB)
// and this block's 16 rows of Q_s (8 KB) come in by bulk async copies into a two-slot shared-memory ring
// while the previous segment is applied: the block waits on memory about once, not once per segment.
// Waits are bounded; on expiry the block latches GDR_ERR_TIMEOUT and stops after its copies in flight
// have landed.
constexpr int SCAN_NT = 128;
constexpr uint32_t SCAN_P = DK * DK * 4, SCAN_Q = 16 * DK * 4, SCAN_SLOT = SCAN_P + SCAN_Q;
constexpr int SCAN_LD = DK + 4;  // row stride of the state rows in shared memory (16-byte aligned rows)
constexpr uint32_t SCAN_S = 2 * SCAN_SLOT, SCAN_BAR = SCAN_S + 16 * SCAN_LD * 4, SCAN_BYTES = SCAN_BAR + 16;
__global__ void __launch_bounds__(SCAN_NT) seg_scan_kernel(int Hv, int nseg, bool reverse, const float *__restrict__ init,
                                                           bool v_first, const float *__restrict__ P,
                                                           const float *__restrict__ Q, float *__restrict__ out,
                                                           unsigned *err, long polls) {
    extern __shared__ __align__(128) unsigned char scan_smem[];
    float *sS = reinterpret_cast<float *>(scan_smem + SCAN_S);  // [16][SCAN_LD]
    const uint32_t sb = smem_u32(scan_smem), bar = sb + SCAN_BAR;
    const int blk = blockIdx.x, j = blockIdx.y, n = blockIdx.z;
    const int tid = threadIdx.x, r0 = (tid >> 5) * 4, c0 = (tid & 31) * 4;
    const long long st_base = ((long long)n * Hv + j) * DK * DV;
    auto seg_base = [&](int t) -> long long {
        const int sg = reverse ? nseg - 1 - t : t;
        return (((long long)n * Hv + j) * nseg + sg) * DK * DV;
    };
    // segment t's P and Q rows into slot t & 1 (thread 0)
    auto fetch = [&](int t) {
        const uint32_t slot = sb + (uint32_t)(t & 1) * SCAN_SLOT, b = bar + 8 * (t & 1);
        const long long sbase = seg_base(t);
        tma::expect_tx(b, SCAN_SLOT);
        for (int i = 0; i < 4; ++i)
            tma::load1d(slot + i * (SCAN_P / 4), P + sbase + i * (DK * DK / 4), SCAN_P / 4, b);
        tma::load1d(slot + SCAN_P, Q + sbase + (long long)blk * 16 * DK, SCAN_Q, b);
    };
    const int steps = nseg - 1;  // segments whose P and Q are applied
    if (tid == 0) {
        umma::mbar_init(bar, 1);
        umma::mbar_init(bar + 8, 1);
        umma::fence_mbar_init();
    }
    for (int r = 0; r < 4; ++r) {
        const int e = blk * 16 + r0 + r;
        for (int c = 0; c < 4; ++c) {
            const int d = c0 + c;
            sS[(r0 + r) * SCAN_LD + d] = init ? init[st_base + (v_first ? (long long)e * DK + d : (long long)d * DV + e)] : 0.f;
        }
    }
    __syncthreads();
    if (tid == 0 && steps > 0) fetch(0);
    int issued = steps > 0 ? 1 : 0;
    bool ok = true;
    for (int t = 0; t < nseg; ++t) {
        const long long sbase = seg_base(t);
        float4 y[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            y[r] = *reinterpret_cast<const float4 *>(sS + (r0 + r) * SCAN_LD + c0);
            *reinterpret_cast<float4 *>(out + sbase + (long long)(blk * 16 + r0 + r) * DK + c0) = y[r];
        }
        if (t >= steps) break;
        // the next segment's copies go into the other slot, which segment t - 1 has finished with
        if (tid == 0 && t + 1 < steps) {
            fetch(t + 1);
            ++issued;
        }
        const bool got = umma::mbar_wait(bar + 8 * (t & 1), (t >> 1) & 1, polls);
        if (__syncthreads_or(!got)) {
            if (tid == 0) raise_error(err, GDR_ERR_TIMEOUT);
            ok = false;
            break;
        }
        const float *sP = reinterpret_cast<const float *>(scan_smem + (t & 1) * SCAN_SLOT);
#pragma unroll
        for (int r = 0; r < 4; ++r) y[r] = *reinterpret_cast<const float4 *>(sP + DK * DK + (r0 + r) * DK + c0);
#pragma unroll 2
        for (int d = 0; d < DK; d += 4) {
            float4 sv[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) sv[r] = *reinterpret_cast<const float4 *>(sS + (r0 + r) * SCAN_LD + d);
#pragma unroll
            for (int dd = 0; dd < 4; ++dd) {
                const float4 pv = *reinterpret_cast<const float4 *>(sP + (d + dd) * DK + c0);
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const float a = dd == 0 ? sv[r].x : dd == 1 ? sv[r].y : dd == 2 ? sv[r].z : sv[r].w;
                    y[r].x += a * pv.x;
                    y[r].y += a * pv.y;
                    y[r].z += a * pv.z;
                    y[r].w += a * pv.w;
                }
            }
        }
        __syncthreads();  // every thread has read S_t and this slot
#pragma unroll
        for (int r = 0; r < 4; ++r) *reinterpret_cast<float4 *>(sS + (r0 + r) * SCAN_LD + c0) = y[r];
        __syncthreads();
    }
    // copies still in flight land before the block exits (bounded)
    if (!ok && tid == 0)
        for (int t = 0; t < issued; ++t) umma::mbar_wait(bar + 8 * (t & 1), (t >> 1) & 1, 4000000L);
}

}  // namespace

namespace {

// dst[b] = src[b]^T for a batch of 128 x 128 fp32 matrices (32 x 32 tiles through shared memory; block x = b,
// block y = the tile).
__global__ void __launch_bounds__(256) transpose128_kernel(const float *__restrict__ src, float *__restrict__ dst) {
    __shared__ float t[32][33];
    const long long base = (long long)blockIdx.x * DK * DK;
    const int r0 = (blockIdx.y >> 2) * 32, c0 = (blockIdx.y & 3) * 32, tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int i = ty; i < 32; i += 8) t[i][tx] = src[base + (long long)(r0 + i) * DK + c0 + tx];
    __syncthreads();
    for (int i = ty; i < 32; i += 8) dst[base + (long long)(c0 + i) * DK + r0 + tx] = t[tx][i];
}

cudaError_t launch_seg_scan(const Args &a, const SegWs &sw, bool reverse, const float *init, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(seg_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SCAN_BYTES);
    if (e != cudaSuccess) return e;
    return launch_plain(seg_scan_kernel, dim3(DV / 16, a.Hv, a.N), dim3(SCAN_NT), SCAN_BYTES, s, a.Hv, sw.nseg,
                        reverse, init, a.v_first, sw.end1, sw.end0, sw.start, a.err,
                        a.wait_polls >= 0 ? (long)a.wait_polls : 200000000L);
}

// [tokens][heads][cols] map with 64 x 1 x 64 boxes
bool tile_map(CUtensorMap *m, const void *base, const Args &a, int heads, int cols) {
    return make_token_map(m, base, a.bf16, cols, heads, (uint64_t)a.B * (uint64_t)a.T, 64);
}

TcBwdP bwd_params(const Args &a, const void *q, const void *k, const float *g_cs, const void *beta, const void *A,
                  const void *dout, const float *dht, void *dhn, void *ddelta, float *dh0, const SegWs &sw) {
    TcBwdP p;
    p.nseg = -1;  // marks a failed tensor-map encoding
    if (!tile_map(&p.tq, q, a, a.Hq, a.K) || !tile_map(&p.tk, k, a, a.Hq, a.K) || !tile_map(&p.tdo, dout, a, a.Hv, a.V) ||
        !tile_map(&p.ta, A, a, a.Hv, C))
        return p;
    p.q = q;
    p.k = k;
    p.A = A;
    p.beta = beta;
    p.dout = dout;
    p.g_cs = g_cs;
    p.dht = dht;
    p.dhn = dhn;
    p.ddelta = ddelta;
    p.dh0 = dh0;
    p.gate_f32 = a.gate_f32;
    p.l2norm = a.l2norm;
    p.v_first = a.v_first;
    p.scale = a.scale;
    p.nseg = sw.nseg;
    p.seg_start = nullptr;
    p.seg_end0 = sw.end0;
    p.seg_end1 = sw.end1;
    return p;
}

TcP fwd_params(const Args &a, const void *q, const void *k, const void *v, const float *g_cs, const void *beta,
               const void *A, const float *h0, void *o, float *final_state, void *h, bool h_api_layout, void *delta,
               const SegWs &sw) {
    TcP p;
    p.nseg = -1;  // marks a failed tensor-map encoding
    if (!tile_map(&p.tq, q, a, a.Hq, a.K) || !tile_map(&p.tk, k, a, a.Hq, a.K) || !tile_map(&p.tv, v, a, a.Hv, a.V) ||
        !tile_map(&p.ta, A, a, a.Hv, C))
        return p;
    p.q = q;
    p.k = k;
    p.v = v;
    p.A = A;
    p.beta = beta;
    p.g_cs = g_cs;
    p.h0 = h0;
    p.o = o;
    p.h = h;
    p.delta = delta;
    p.fin = final_state;
    p.gate_f32 = a.gate_f32;
    p.l2norm = a.l2norm;
    p.v_first = a.v_first;
    p.h_api = h_api_layout;
    p.scale = a.scale;
    p.nseg = sw.nseg;
    p.seg_start = nullptr;
    p.seg_end0 = sw.end0;
    p.seg_end1 = sw.end1;
    return p;
}

}  // namespace

cudaError_t launch_chain_bwd_affine(const Args &a, const void *q, const void *k, const float *g_cs, const void *beta,
                                    const void *A, const void *dout, const float *dht, const SegWs &sw, cudaStream_t s) {
    if (sw.nseg < 2) return cudaErrorInvalidValue;
    TcBwdP p = bwd_params(a, q, k, g_cs, beta, A, dout, dht, nullptr, nullptr, nullptr, sw);
    if (p.nseg < 1) return cudaErrorInvalidValue;
    cudaError_t e = a.bf16 ? chain_bwd_tc_t<__nv_bfloat16>(a, p, true, s) : chain_bwd_tc_t<__half>(a, p, true, s);
    if (e != cudaSuccess) return e;
    return launch_seg_scan(a, sw, true, dht, s);
}

cudaError_t launch_fwd_compose(const Args &a, const float *h0, const SegWs &sw, cudaStream_t s) {
    if (sw.nseg < 2) return cudaErrorInvalidValue;
    return launch_seg_scan(a, sw, false, h0, s);
}

// The reverse chain is the adjoint of the forward's linear part: a segment's transfer matrix for the reverse
// scan is the transpose of the forward's.
cudaError_t launch_rev_compose(const Args &a, const float *dht, const float *fwd_transfer, const SegWs &sw,
                               cudaStream_t s) {
    if (sw.nseg < 2 || !fwd_transfer) return cudaErrorInvalidValue;
    cudaError_t e = launch_plain(transpose128_kernel, dim3((unsigned)((long long)a.N * a.Hv * sw.nseg), 16), dim3(256),
                                 0, s, fwd_transfer, sw.end1);
    if (e != cudaSuccess) return e;
    return launch_seg_scan(a, sw, true, dht, s);
}

cudaError_t launch_chain_bwd(const Args &a, const void *q, const void *k, const float *g_cs, const void *beta,
                             const void *A, const void *dout, const float *dht, void *dhn, void *ddelta, float *dh0,
                             const SegWs &sw, cudaStream_t s) {
    TcBwdP p = bwd_params(a, q, k, g_cs, beta, A, dout, dht, dhn, ddelta, dh0, sw);
    if (p.nseg < 1) return cudaErrorInvalidValue;
    cudaError_t e;
    if (sw.nseg > 1) {
        if ((e = launch_chain_bwd_affine(a, q, k, g_cs, beta, A, dout, dht, sw, s)) != cudaSuccess) return e;
        p.seg_start = sw.start;
    }
    return a.bf16 ? chain_bwd_tc_t<__nv_bfloat16>(a, p, false, s) : chain_bwd_tc_t<__half>(a, p, false, s);
}

cudaError_t launch_chain_fwd_affine(const Args &a, const void *q, const void *k, const void *v, const float *g_cs,
                                    const void *beta, const void *A, const float *h0, const SegWs &sw, cudaStream_t s) {
    if (sw.nseg < 2) return cudaErrorInvalidValue;
    TcP p = fwd_params(a, q, k, v, g_cs, beta, A, h0, nullptr, nullptr, nullptr, false, nullptr, sw);
    if (p.nseg < 1) return cudaErrorInvalidValue;
    cudaError_t e =
        a.bf16 ? chain_fwd_tc_t<__nv_bfloat16>(a, p, false, true, s) : chain_fwd_tc_t<__half>(a, p, false, true, s);
    if (e != cudaSuccess) return e;
    return launch_seg_scan(a, sw, false, h0, s);
}

cudaError_t launch_chain_fwd(const Args &a, const void *q, const void *k, const void *v, const float *g_cs,
                             const void *beta, const void *A, const float *h0, void *o, float *final_state, void *h,
                             bool h_api_layout, void *delta, const SegWs &sw, cudaStream_t s) {
    TcP p = fwd_params(a, q, k, v, g_cs, beta, A, h0, o, final_state, h, h_api_layout, delta, sw);
    if (p.nseg < 1) return cudaErrorInvalidValue;
    cudaError_t e;
    if (sw.nseg > 1) {
        if ((e = launch_chain_fwd_affine(a, q, k, v, g_cs, beta, A, h0, sw, s)) != cudaSuccess) return e;
        p.seg_start = sw.start;
    }
    return a.bf16 ? chain_fwd_tc_t<__nv_bfloat16>(a, p, o != nullptr, false, s)
                  : chain_fwd_tc_t<__half>(a, p, o != nullptr, false, s);
}

}  // namespace gdr
