// The state-independent per-chunk work of the forward, on tcgen05 (FlashQLA skill page, "Low-Level API": the
// forward returns the processed gate and the intra-chunk matrix A; the chunk form of the recurrence in the
// "Core API" section): for every chunk and value head, with G the chunk-local cumsum of the log-gate,
// Gamma_rs = exp(G_r - G_s) and q^ = nq q, k^ = nk k the (optionally) L2-normalised rows,
//
//   g_cumsum = G
//   L = strictly-lower(diag(beta) (k^ k^^T o Gamma)),   A = (I + L)^-1
//   P = scale (q^ k^^T o Gamma) for s <= r (zero above the diagonal)   -- the decayed causal block
//   nq, nk                                                               -- the inverse row norms
//
// Persistent CTAs of 128 threads (four per SM) walk (chunk, q/k head) items; the value heads of the item's
// GVA group reuse its one product.  The q and k tiles of an item arrive by TMA; the other CTAs on the SM
// cover each one's load and MMA latency.  One MMA computes [Q;K] K^T (M = 128, N = 64, K = 128): TMEM lanes
// 0..63 hold Q K^T (the P rows, epilogue of warps 0 and 1) and lanes 64..127 hold K K^T (the L rows, warps 2
// and 3).  The decays enter as 2^(G_r log2 e - LG_s) with the column table LG_s = G_s log2 e - log2 nk_s, so
// no factor e^{-G} is ever formed on its own.  The inverse of the unit lower-triangular I + L: the four
// 16 x 16 diagonal blocks by substitution in fp32 on the CUDA cores, then the off-diagonal blocks by block
// distance (1, 2, 3), A_ij = -A_ii sum_{k=j}^{i-1} L_ik A_kj, with warp-level tf32 MMAs on 16 x 8 pieces.
// Full chunks' P rows leave through a swizzled staging tile and a TMA store, A rows by coalesced stores; a
// ragged chunk's rows are stored directly (its tail rows belong to the next sequence).
#include <cuda_runtime.h>

#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tmap.h"
#include "umma.cuh"

namespace gdr {
namespace {

constexpr int WT = 128;
template <typename T> struct IsBf16 { static constexpr bool value = false; };
template <> struct IsBf16<__nv_bfloat16> { static constexpr bool value = true; };

// ---- shared memory (bytes from a 1024-aligned base).  The stage region first holds the q and k tiles of the
// item, [Q b0][K b0][Q b1][K b1] in 8 KB blocks; once the MMA has read them (and the row norms are taken) it
// holds L and A^-1 in fp32, 64 x 64 each with rows of LDF floats (4 mod 32: a warp's row-per-thread float4
// stores and its fragment loads are conflict-free).  Four CTAs per SM hide each other's load and MMA latencies.
constexpr uint32_t ST_BYTES = 32768;
constexpr int LDF = 68;
constexpr uint32_t MAT_BYTES = 64 * LDF * 4;
constexpr uint32_t S_L = 0, S_AI = MAT_BYTES;        // over the stage
constexpr uint32_t S_PST = 36864;                    // P staging tile, 64 x 64 16-bit, swizzled
static_assert(2 * MAT_BYTES <= S_PST && ST_BYTES <= S_PST, "stage region");
constexpr int LDS_ = 9;                              // row stride of a warp's 16 x 8 merge scratch
constexpr uint32_t S_W = S_PST + 8192;               // merge scratch, one 16 x 8 fp32 block per warp
constexpr uint32_t S_SC = S_W + 4 * 16 * LDS_ * 4;
// 64 floats each: nq, nk (inverse norms), G, LG (G log2 e - log2 nk), BQ (scale nq), BL (beta nk), GT (scan carry)
enum { F_NQ = 0, F_NK, F_G, F_LG, F_BQ, F_BL, F_GT, F_COUNT };
constexpr uint32_t S_RING = S_SC + F_COUNT * 256;    // the item being loaded: {first token, valid rows, q/k head, -}
constexpr uint32_t S_BAR = S_RING + 16;              // full, mma
constexpr uint32_t S_SLOT = S_BAR + 16, S_FLAG = S_SLOT + 4;
constexpr uint32_t S_BYTES = S_FLAG + 4 + 1024;
static_assert(S_BAR % 8 == 0 && S_SC % 16 == 0, "alignment");
static_assert(4 * (S_BYTES + 1024) <= 233472, "four CTAs per SM");
constexpr uint32_t T_COLS = 64;
constexpr uint32_t TILE_BYTES = ST_BYTES;
constexpr float LOG2E = 1.4426950408889634f;

struct WyP {
    CUtensorMap tq, tk, tp;      // q, k [tokens][Hq][K]; P [tokens][Hv][64]; boxes 64 x 1 x 64
    const void *g, *beta;        // raw log-gate and beta [tokens][Hv] (element type or fp32)
    float *g_cs;                 // out: [tokens][Hv]
    void *P, *A;                 // out: [tokens][Hv][64] (P may be null)
    float *rq, *rk;              // out: inverse norms [tokens][Hv] (null unless requested)
    bool gate_f32, l2norm;
    float scale;
    int nslots;
    long polls;
};

// 2^x in one MUFU instruction (flushes subnormal results to zero; the decays here need no subnormals).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// One 16 x 8 piece of an off-diagonal block of A = (I + L)^-1 at block distance LV (block row i = LV + q,
// block column j = q, columns n0 .. n0 + 7 with n0 = 16 j + 8 nt), by one warp with tf32 tensor-core MMAs
// (m16n8k8; the 16 x 16 blocks are a quarter of tcgen05's smallest tile):
//   R = sum_{k = 16 j}^{16 i - 1} L[16 i .., k] A[k, n0 ..]        (every A block used is already known)
//   A[16 i .., n0 ..] = -A_ii R
// R goes through the warp's scratch to change from accumulator to B-operand layout.
__device__ __forceinline__ void merge_piece(int LV, int q, int nt, const float *L, float *Ai, float *scr, int lane) {
    const int g = lane >> 2, t = lane & 3;
    const int i = LV + q, j = q, n0 = 16 * j + 8 * nt, r0 = 16 * i;
    float r[4] = {0.f, 0.f, 0.f, 0.f};
    for (int kk = 0; kk < 2 * LV; ++kk) {
        const int kc = 16 * j + 8 * kk;
        uint32_t a[4];
        a[0] = to_tf32(L[(r0 + g) * LDF + kc + t]);
        a[1] = to_tf32(L[(r0 + g + 8) * LDF + kc + t]);
        a[2] = to_tf32(L[(r0 + g) * LDF + kc + t + 4]);
        a[3] = to_tf32(L[(r0 + g + 8) * LDF + kc + t + 4]);
        const uint32_t b0 = to_tf32(Ai[(kc + t) * LDF + n0 + g]);
        const uint32_t b1 = to_tf32(Ai[(kc + t + 4) * LDF + n0 + g]);
        mma1688_tf32(r, a, b0, b1);
    }
    scr[g * LDS_ + 2 * t] = r[0];
    scr[g * LDS_ + 2 * t + 1] = r[1];
    scr[(g + 8) * LDS_ + 2 * t] = r[2];
    scr[(g + 8) * LDS_ + 2 * t + 1] = r[3];
    __syncwarp();
    float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
        const int kc = r0 + 8 * kk;
        uint32_t a[4];
        a[0] = to_tf32(Ai[(r0 + g) * LDF + kc + t]);
        a[1] = to_tf32(Ai[(r0 + g + 8) * LDF + kc + t]);
        a[2] = to_tf32(Ai[(r0 + g) * LDF + kc + t + 4]);
        a[3] = to_tf32(Ai[(r0 + g + 8) * LDF + kc + t + 4]);
        const uint32_t b0 = to_tf32(scr[(8 * kk + t) * LDS_ + g]);
        const uint32_t b1 = to_tf32(scr[(8 * kk + t + 4) * LDS_ + g]);
        mma1688_tf32(o, a, b0, b1);
    }
    Ai[(r0 + g) * LDF + n0 + 2 * t] = -o[0];
    Ai[(r0 + g) * LDF + n0 + 2 * t + 1] = -o[1];
    Ai[(r0 + g + 8) * LDF + n0 + 2 * t] = -o[2];
    Ai[(r0 + g + 8) * LDF + n0 + 2 * t + 1] = -o[3];
    __syncwarp();
}

template <typename T>
__global__ void __launch_bounds__(WT, 4) wy_tc_kernel(Geo geo, const __grid_constant__ WyP p) {
    griddep_launch_next();
    griddep_wait();
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const int Hv = geo.Hv, Hq = geo.Hq, grp = Hv / Hq;
    const int nitems = p.nslots * Hq;  // the host keeps this below 2^31
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float *F = reinterpret_cast<float *>(smem + S_SC);
    auto fs = [&](int slot, int i) -> float & { return F[slot * 64 + i]; };
    float *Lm = reinterpret_cast<float *>(smem + S_L);
    float *Ai = reinterpret_cast<float *>(smem + S_AI);
    int4 *ring = reinterpret_cast<int4 *>(smem + S_RING);
    volatile int *sflag = reinterpret_cast<volatile int *>(smem + S_FLAG);
    const uint32_t full = sb + S_BAR, mbar = sb + S_BAR + 8;
    const bool want_p = p.P != nullptr;

    if (tid == 0) {
        umma::mbar_init(full, 1);
        umma::mbar_init(mbar, 1);
        umma::fence_mbar_init();
        *sflag = 0;
    }
    if (warp == 0) umma::alloc(sb + S_SLOT, T_COLS);
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + S_SLOT);
    constexpr bool bf16 = IsBf16<T>::value;
    const uint32_t i_n64 = umma::idesc(128, 64, bf16, false, false);

    // ---- the item walk (thread 0): w = blockIdx.x, + gridDim.x, ... skipping empty varlen slots; the item's
    //      place goes to the ring slot (valid = -1: none left) and its tiles into the stage
    int wiss = (int)blockIdx.x;
    int loads = 0, seen = 0;  // thread 0: loads issued / completions seen
    auto produce = [&]() {
        int4 u = make_int4(0, -1, 0, 0);
        for (; wiss < nitems; wiss += (int)gridDim.x) {
            const int slot_ = geo.div_hq(wiss);
            long long t_;
            int n_, c_, v_;
            if (geo.chunk(slot_, t_, v_, n_, c_)) {
                u = make_int4((int)t_, v_, wiss - slot_ * Hq, 0);
                wiss += (int)gridDim.x;
                break;
            }
        }
        ring[0] = u;
        if (u.y < 0) return;
        ++loads;
        tma::expect_tx(full, TILE_BYTES);
        tma::load3d(sb, &p.tq, 0, u.z, u.x, full);
        tma::load3d(sb + 8192, &p.tk, 0, u.z, u.x, full);
        tma::load3d(sb + 16384, &p.tq, 64, u.z, u.x, full);
        tma::load3d(sb + 24576, &p.tk, 64, u.z, u.x, full);
    };
    if (tid == 0) produce();
    __syncthreads();

    // gates of (item u, value head j) for rows 0..63 (threads 0..63), fetched one step ahead as predicated
    // loads that nothing reads before the step that uses them
    // A log-gate below kGateFloor is taken at kGateFloor: its decay factor e^g (< 2e-35) already wipes the
    // state at fp32 resolution, and the chunk form subtracts cumulative gates, which a gate of -inf (a hard
    // reset) would turn into -inf - (-inf).  NaN gates pass through.
    constexpr float kGateFloor = -80.f;
    float gnext = 0.f, bnext = 0.f;
    auto fetch_g = [&](const int4 &u, int j_) {
        gnext = 0.f;
        bnext = 0.f;
        if (tid < u.y && tid < C) {
            const long long ti = ((long long)u.x + tid) * Hv + j_;
            gnext = load_gate<T>(p.g, ti, p.gate_f32);
            if (gnext < kGateFloor) gnext = kGateFloor;
            bnext = load_gate<T>(p.beta, ti, p.gate_f32);
        }
    };
    int4 cur = ring[0];
    if (cur.y >= 0) fetch_g(cur, cur.z * grp);
    uint32_t fph = 0, mph = 0;  // thread 0: the phase to wait for on the full barrier and on mbar
    bool mma_out = false;       // thread 0: an MMA whose completion was not seen
    const int r = tid & 63;     // the row of this thread's TMEM lane (Q rows: warps 0, 1; K rows: warps 2, 3)
    const bool krow = tid >= 64;

    while (cur.y >= 0) {
        const int valid = cur.y;
        if (tid == 0) {
            if (umma::mbar_spin(full, fph, p.polls)) {
                fph ^= 1u;
                ++seen;
            } else {
                raise_error(geo.err, GDR_ERR_TIMEOUT);
                *sflag = 1;
            }
        }
        umma::fence_before();
        __syncthreads();
        umma::fence_after();
        if (*sflag) break;
        // [Q;K] K^T (K = 128 in eight steps of 16)
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t ko = (uint32_t)(ks >> 2) * 16384u + (uint32_t)(ks & 3) * 32u;
                umma::mma(tmem, umma::desc(sb + ko, 16, 1024), umma::desc(sb + 8192 + ko, 16, 1024), i_n64, ks > 0);
            }
            umma::commit(mbar);
            mma_out = true;
        }
        // meanwhile the inverse row norms: thread t < 64 takes q row t, thread 64 + t k row t
        if (p.l2norm) {
            const uint32_t base = sb + (krow ? 8192u : 0u);
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const uint4 u = umma::ld_shared_v4(base + (uint32_t)(c >> 3) * 16384u + umma::off(r, (c & 7) * 8, 0));
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 x = Elt<T>::unpack(w[e]);
                    s0 = fmaf(x.x, x.x, s0);
                    s1 = fmaf(x.y, x.y, s1);
                }
            }
            fs(krow ? F_NK : F_NQ, r) = 1.0f / sqrtf(s0 + s1 + L2_EPS);
        } else {
            fs(krow ? F_NK : F_NQ, r) = 1.f;
        }
        if (tid == 0) {
            if (umma::mbar_spin(mbar, mph, p.polls)) {
                mph ^= 1u;
                mma_out = false;
            } else {
                raise_error(geo.err, GDR_ERR_TIMEOUT);
                *sflag = 1;
            }
        }
        umma::fence_before();
        __syncthreads();
        umma::fence_after();
        if (*sflag) break;
        const bool staged = valid == C;

        for (int jj = 0; jj < grp; ++jj) {
            const int j = cur.z * grp + jj;
            // ---- gates: chunk-local inclusive cumsum of g over rows 0..63 (warps 0 and 1), beta
            if (tid == 0) tma::wait_read();  // the previous P tile has left its staging buffer
            float gv = gnext, bv = bnext;
            if (jj + 1 < grp) fetch_g(cur, j + 1);  // the next value head's gates, while this one works
            if (tid < C) {
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, gv, o);
                    if (lane >= o) gv += y;
                }
                if (tid == 31) fs(F_GT, 0) = gv;
            }
            __syncthreads();
            if (tid < C) {
                if (tid >= 32) gv += fs(F_GT, 0);
                fs(F_G, tid) = gv;
                fs(F_LG, tid) = gv * LOG2E - log2f(fs(F_NK, tid));
                fs(F_BQ, tid) = p.scale * fs(F_NQ, tid);
                fs(F_BL, tid) = bv * fs(F_NK, tid);
                if (tid < valid) p.g_cs[((long long)cur.x + tid) * Hv + j] = gv;
            }
            __syncthreads();
            // ---- epilogue: P rows (warps 0, 1) and L rows (warps 2, 3), 64 columns per thread in four steps of
            //      16; P_rs = BQ_r 2^(G_r log2 e - LG_s) (Q K^T)_rs, L_rs = BL_r 2^(G_r log2 e - LG_s) (K K^T)_rs.
            //      Rows 0..31 (warps 0 and 2) have nothing right of column 31.
            {
                const float gr2 = fs(F_G, r) * LOG2E;
                const float rf = krow ? fs(F_BL, r) : fs(F_BQ, r);
                const bool rv = r < valid;
                const int nh = (warp & 1) ? 4 : 2;  // column steps that can hold nonzeros
                const float4 *lg4 = reinterpret_cast<const float4 *>(&fs(F_LG, 0));
                if (krow) {
                    float4 *lrow = reinterpret_cast<float4 *>(Lm + r * LDF);
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        if (h < nh) {
                            float x[16];
                            umma::ld16(umma::taddr(tmem, warp * 32, h * 16), x);
                            umma::ld_wait();
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const float4 l = lg4[4 * h + u];
                                const float lv[4] = {l.x, l.y, l.z, l.w};
                                float v[4];
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const int s = h * 16 + 4 * u + e;
                                    const float y = ex2(gr2 - lv[e]) * x[4 * u + e] * rf;
                                    v[e] = (s < r && rv) ? y : 0.f;
                                }
                                lrow[4 * h + u] = make_float4(v[0], v[1], v[2], v[3]);
                            }
                        } else {
#pragma unroll
                            for (int u = 0; u < 4; ++u) lrow[4 * h + u] = make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                    }
                    if (p.rk && p.l2norm && rv) p.rk[((long long)cur.x + r) * Hv + j] = fs(F_NK, r);
                } else if (want_p) {
                    T *dst = static_cast<T *>(p.P) + (((long long)cur.x + r) * Hv + j) * C;
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        uint32_t w[8];
                        if (h < nh) {
                            float x[16];
                            umma::ld16(umma::taddr(tmem, warp * 32, h * 16), x);
                            umma::ld_wait();
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const float4 l = lg4[4 * h + u];
                                const float lv[4] = {l.x, l.y, l.z, l.w};
                                float v[4];
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const int s = h * 16 + 4 * u + e;
                                    const float y = ex2(gr2 - lv[e]) * x[4 * u + e] * rf;
                                    v[e] = (s <= r && rv) ? y : 0.f;
                                }
                                w[2 * u] = Elt<T>::pack(v[0], v[1]);
                                w[2 * u + 1] = Elt<T>::pack(v[2], v[3]);
                            }
                        } else {
#pragma unroll
                            for (int u = 0; u < 8; ++u) w[u] = 0u;
                        }
                        if (staged) {
#pragma unroll
                            for (int c = 0; c < 2; ++c)
                                umma::st_shared_v4(sb + S_PST + umma::off(r, h * 16 + c * 8, 0), w[4 * c], w[4 * c + 1],
                                                   w[4 * c + 2], w[4 * c + 3]);
                        } else if (rv) {
#pragma unroll
                            for (int c = 0; c < 2; ++c)
                                *reinterpret_cast<uint4 *>(dst + h * 16 + c * 8) =
                                    make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
                        }
                    }
                    if (p.rq && p.l2norm && rv) p.rq[((long long)cur.x + r) * Hv + j] = fs(F_NQ, r);
                }
            }
            if (staged && want_p) umma::fence_async_smem();
            // the item's last head: TMEM is read out, so the next item's place and gates can be looked up
            umma::fence_before();
            __syncthreads();
            if (tid == 0 && staged && want_p) {
                tma::store3d(&p.tp, 0, j, cur.x, sb + S_PST);
                tma::commit_group();
            }
            // ---- diagonal 16 x 16 blocks of (I + L)^-1 in fp32: warp w takes block w, lane c < 16 its column c,
            //      by forward substitution with right-looking updates (one dependent step per row)
            if (lane < 16) {
                const int b0 = warp * 16;
                const float *lb = Lm + b0 * LDF + b0;
                float acc[16], x[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[i] = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    x[i] = (i == lane) ? 1.f : (i > lane ? acc[i] : 0.f);
#pragma unroll
                    for (int k = i + 1; k < 16; ++k) acc[k] = fmaf(-lb[k * LDF + i], x[i], acc[k]);
                }
                float *ab = Ai + b0 * LDF + b0 + lane;
#pragma unroll
                for (int i = 0; i < 16; ++i) ab[i * LDF] = x[i];
            }
            __syncthreads();
            // ---- off-diagonal blocks by block distance: six, four and two 16 x 8 pieces over the four warps
            {
                float *scr = reinterpret_cast<float *>(smem + S_W) + warp * 16 * LDS_;
                merge_piece(1, warp >> 1, warp & 1, Lm, Ai, scr, lane);
                if (warp < 2) merge_piece(1, 2, warp, Lm, Ai, scr, lane);
                __syncthreads();
                merge_piece(2, warp >> 1, warp & 1, Lm, Ai, scr, lane);
                __syncthreads();
                if (warp < 2) merge_piece(3, 0, warp, Lm, Ai, scr, lane);
                __syncthreads();
            }
            // ---- A out: row r of the chunk at token cur.x + r, zero above the diagonal (coalesced rows)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int id = tid + WT * u, row = id >> 3, c8 = id & 7;
                if (row < valid) {
                    const float4 a0 = *reinterpret_cast<const float4 *>(Ai + row * LDF + 8 * c8);
                    const float4 a1 = *reinterpret_cast<const float4 *>(Ai + row * LDF + 8 * c8 + 4);
                    const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int c = 8 * c8 + 2 * e;
                        w[e] = Elt<T>::pack(c <= row ? av[2 * e] : 0.f, c + 1 <= row ? av[2 * e + 1] : 0.f);
                    }
                    *reinterpret_cast<uint4 *>(static_cast<T *>(p.A) + (((long long)cur.x + row) * Hv + j) * C + 8 * c8) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            umma::fence_async_smem();  // (the stage's next writer is the async proxy)
            __syncthreads();
        }
        // L and A^-1 are read: the stage takes the next item's tiles; TMEM is free for its MMA
        if (tid == 0) produce();
        umma::fence_before();
        __syncthreads();
        umma::fence_after();
        cur = ring[0];
        if (cur.y >= 0) fetch_g(cur, cur.z * grp);
    }
    // after an error, let the load and the MMA in flight finish before the block exits (bounded waits);
    // the P stores complete before shared memory goes away
    if (tid == 0) {
        if (loads > seen) umma::mbar_wait(full, fph, 4000000L);
        if (mma_out) umma::mbar_wait(mbar, mph, 4000000L);
        tma::wait_all();
    }
    umma::fence_before();
    __syncthreads();
    if (warp == 0) umma::dealloc(tmem, T_COLS);
}

template <typename T>
cudaError_t wy_tc_t(const Args &a, const WyP &p, cudaStream_t s) {
    if (a.max_chunks == 0) return cudaSuccess;
    if ((long long)a.max_chunks * a.Hq >= (1ll << 31)) return cudaErrorInvalidValue;  // 32-bit item indices
    auto kern = wy_tc_kernel<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S_BYTES);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const long items = (long)a.max_chunks * a.Hq;
    const unsigned grid = (unsigned)(items < 4L * sms ? items : 4L * sms);  // four persistent CTAs per SM
    return launch_overlapped(kern, dim3(grid), dim3(WT), S_BYTES, s, make_geo(a), p);
}

}  // namespace

cudaError_t launch_wy_fwd(const Args &a, const void *q, const void *k, const void *g, const void *beta, float *g_cs,
                          void *A, void *P, float *rq, float *rk, cudaStream_t s) {
    WyP p;
    const uint64_t tokens = (uint64_t)a.B * (uint64_t)a.T;
    const bool bf = a.bf16;
    if (!make_token_map(&p.tq, q, bf, a.K, a.Hq, tokens, 64) || !make_token_map(&p.tk, k, bf, a.K, a.Hq, tokens, 64))
        return cudaErrorInvalidValue;
    if (P && !make_tmap_3d(&p.tp, P, bf, C, a.Hv, tokens, C * 2, (uint64_t)a.Hv * C * 2, 64, 1, 64))
        return cudaErrorInvalidValue;
    p.g = g;
    p.beta = beta;
    p.g_cs = g_cs;
    p.P = P;
    p.A = A;
    p.rq = rq;
    p.rk = rk;
    p.gate_f32 = a.gate_f32;
    p.l2norm = a.l2norm;
    p.scale = a.scale;
    p.nslots = (int)a.max_chunks;
    p.polls = a.wait_polls >= 0 ? (long)a.wait_polls : 200000000L;
    return a.bf16 ? wy_tc_t<__nv_bfloat16>(a, p, s) : wy_tc_t<__half>(a, p, s);
}

}  // namespace gdr
