// The decayed causal block of every chunk and value head for the backward's chains, on tcgen05:
//   P = scale (q^ k^^T o Gamma), s <= r < valid (zero elsewhere),  Gamma_rs = exp(G_r - G_s),
// with G the chunk-local gate cumsum, q^ = nq q and k^ = nk k the L2-normalised rows (nq = nk = 1 without
// normalisation), and the inverse norms nq, nk themselves (FlashQLA skill page, "Low-Level API": the
// backward takes g_cumsum from the forward; the decayed block is the intra-chunk attention term of the
// chunked form).
//
// Two persistent CTAs of 128 threads per SM walk (chunk, q/k head) items.  Each item's q and k tiles arrive
// by TMA into one of two stages (the next item's tiles land while one is processed; the other CTA on the SM
// covers this one's latencies); one MMA computes
// [Q;Q] K^T, so TMEM lanes r and 64 + r both hold row r of Q K^T and all four warps share the epilogue
// (lanes 0..63 columns 0..31, lanes 64..127 columns 32..63).  The rows of a full chunk leave through a
// swizzled staging tile and a TMA store; a ragged chunk's rows are stored directly (its tail rows belong
// to the next sequence).  The item's value heads (GVA groups) reuse the one product with their own gates.
#include <cuda_runtime.h>

#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tmap.h"
#include "umma.cuh"

namespace gdr {
namespace {

constexpr int PT = 128;
template <typename T> struct IsBf16 { static constexpr bool value = false; };
template <> struct IsBf16<__nv_bfloat16> { static constexpr bool value = true; };
// ---- shared memory (bytes from a 1024-aligned base).  Stage s at s * ST_BYTES: [Q b0][Q b0][Q b1][Q b1]
// (each 64-column block of Q twice: the K-major M=128 operand [Q;Q]) and [K b0][K b1].
constexpr int NST = 2;
constexpr uint32_t ST_BYTES = 49152, ST_Q = 0, ST_K = 32768;
constexpr uint32_t S_PST = NST * ST_BYTES;  // P staging tile [64 x 64]
// 64 floats each: nq, nk (inverse norms), G (gates), LG (G log2 e - log2 nk: the column factor in exp2 form)
constexpr uint32_t S_NQ = S_PST + 8192, S_NK = S_NQ + 256, S_G = S_NK + 256, S_LG = S_G + 256;
constexpr uint32_t S_RING = S_LG + 256;         // per stage: the item's {first token, valid rows, q/k head, -}
constexpr uint32_t S_CNT = S_RING + 16 * NST;   // per stage: loads issued (producer), loads seen (thread 0)
constexpr uint32_t S_BAR = S_CNT + 8 * NST;     // full[NST], mma
constexpr uint32_t S_SLOT = S_BAR + 8 * NST + 8, S_FLAG = S_SLOT + 4;
constexpr uint32_t S_BYTES = S_FLAG + 4 + 1024;
constexpr uint32_t T_COLS = 64;
constexpr uint32_t TILE_BYTES = 49152;  // bytes one item's loads bring in
constexpr int PR = 64;  // the producer thread (warp 2: its rows 0..31 x columns 32..63 of P are all zero)

struct PpP {
    CUtensorMap tq, tk, tp;  // q, k [tokens][Hq][K]; P [tokens][Hv][64]; boxes 64 x 1 x 64
    const float *g_cs;
    void *P;
    float *rq, *rk;
    bool l2norm;
    float scale;
    int nslots;
    long polls;  // bound of the two waits of the item loop
};

template <typename T>
__global__ void __launch_bounds__(PT, 2) chunk_p_tc_kernel(Geo geo, const __grid_constant__ PpP p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const int Hv = geo.Hv, Hq = geo.Hq, grp = Hv / Hq;
    const int nitems = p.nslots * Hq;  // the host keeps this below 2^31
    const int tid = threadIdx.x, warp = tid >> 5;
    const int r = tid & 63, half = tid >> 6;  // row of this thread's TMEM lane, column half of the epilogue
    float *nq = reinterpret_cast<float *>(smem + S_NQ);
    float *nk = reinterpret_cast<float *>(smem + S_NK);
    float *sg = reinterpret_cast<float *>(smem + S_G);
    float *lg = reinterpret_cast<float *>(smem + S_LG);
    int4 *ring = reinterpret_cast<int4 *>(smem + S_RING);
    int *iss = reinterpret_cast<int *>(smem + S_CNT), *seen = iss + NST;
    volatile int *sflag = reinterpret_cast<volatile int *>(smem + S_FLAG);
    const uint32_t full0 = sb + S_BAR, mbar = sb + S_BAR + 8 * NST;

    if (tid == 0) {
        for (int sx = 0; sx < NST; ++sx) {
            umma::mbar_init(full0 + 8u * (uint32_t)sx, 1);
            iss[sx] = 0;
            seen[sx] = 0;
        }
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

    // ---- the producer's item walk: w = blockIdx.x, + gridDim.x, ... (skipping empty varlen slots); it
    //      writes each item's place into the ring slot of the stage the item loads into (valid = -1: none)
    int wiss = (int)blockIdx.x;
    auto produce = [&](int stage) {
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
        ring[stage] = u;
        if (u.y < 0) return;
        const uint32_t st = sb + (uint32_t)stage * ST_BYTES, bar = full0 + 8u * (uint32_t)stage;
        iss[stage] += 1;
        tma::expect_tx(bar, TILE_BYTES);
        tma::load3d(st + ST_Q, &p.tq, 0, u.z, u.x, bar);
        tma::load3d(st + ST_Q + 8192, &p.tq, 0, u.z, u.x, bar);
        tma::load3d(st + ST_Q + 16384, &p.tq, 64, u.z, u.x, bar);
        tma::load3d(st + ST_Q + 24576, &p.tq, 64, u.z, u.x, bar);
        tma::load3d(st + ST_K, &p.tk, 0, u.z, u.x, bar);
        tma::load3d(st + ST_K + 8192, &p.tk, 64, u.z, u.x, bar);
    };
    if (tid == PR)
        for (int sx = 0; sx < NST; ++sx) produce(sx);
    __syncthreads();

    // gates of (item u, value head j) for rows 0..63 (threads 0..63), fetched one step ahead as predicated
    // loads that nothing reads before the step that uses them
    float gnext = 0.f;
    auto fetch_g = [&](const int4 &u, int j_) {
        gnext = 0.f;
        if (tid < u.y) gnext = p.g_cs[((long long)u.x + tid) * Hv + j_];
    };
    int stage = 0;
    int4 cur = ring[0];
    if (cur.y >= 0) fetch_g(cur, cur.z * grp);
    uint32_t fph = 0, mph = 0;  // thread 0: the phase to wait for on each full barrier (bit s) and on mbar
    bool mma_out = false;       // thread 0: an MMA whose completion was not seen

    while (cur.y >= 0) {
        const uint32_t st = sb + (uint32_t)stage * ST_BYTES;
        if (tid == 0) {
            if (umma::mbar_spin(full0 + 8u * (uint32_t)stage, (fph >> stage) & 1u, p.polls)) {
                fph ^= 1u << stage;
                seen[stage] += 1;
            } else {
                raise_error(geo.err, GDR_ERR_TIMEOUT);
                *sflag = 1;
            }
        }
        umma::fence_before();
        __syncthreads();
        umma::fence_after();
        if (*sflag) break;
        // [Q;Q] K^T (K = 128 in eight steps of 16)
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint64_t a = umma::desc(st + ST_Q + (uint32_t)(ks >> 2) * 16384u + (uint32_t)(ks & 3) * 32u, 16, 1024);
                const uint64_t b = umma::desc(st + ST_K + (uint32_t)(ks >> 2) * 8192u + (uint32_t)(ks & 3) * 32u, 16, 1024);
                umma::mma(tmem, a, b, i_n64, ks > 0);
            }
            umma::commit(mbar);
            mma_out = true;
        }
        // meanwhile the row norms: thread t < 64 takes q row t, thread 64 + t k row t (16-byte chunks in the
        // same order on eight consecutive rows: eight distinct bank groups)
        if (p.l2norm) {
            const uint32_t base = st + (half ? ST_K : ST_Q), bstride = half ? 8192u : 16384u;
            float ss = 0.f;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const uint4 u = umma::ld_shared_v4(base + (uint32_t)(c >> 3) * bstride + umma::off(r, (c & 7) * 8, 0));
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 x = Elt<T>::unpack(w[e]);
                    ss += x.x * x.x + x.y * x.y;
                }
            }
            (half ? nk : nq)[r] = 1.0f / sqrtf(ss + L2_EPS);
        } else {
            (half ? nk : nq)[r] = 1.f;
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
        const int4 nxt = ring[stage == NST - 1 ? 0 : stage + 1];  // the next item (written NST - 1 items ago)
        // the stage's tiles have been read (MMA complete, norms taken): the item NST ahead may load into it
        if (tid == PR) produce(stage);
        // this thread's 32 products of row r (TMEM lanes 32 warp.., columns 32 half..); warp 2's block
        // (rows 0..31, columns 32..63) lies above the diagonal
        const bool zero_blk = warp == 2;
        float x[32];
        if (!zero_blk) {
            umma::ld16(umma::taddr(tmem, warp * 32, half * 32), x);
            umma::ld16(umma::taddr(tmem, warp * 32, half * 32 + 16), x + 16);
            umma::ld_wait();
            const float rs = p.scale * nq[r];
#pragma unroll
            for (int u = 0; u < 32; ++u) x[u] *= rs;
        }
        const bool staged = cur.y == C;
        constexpr float LOG2E = 1.4426950408889634f;
        for (int jj = 0; jj < grp; ++jj) {
            const int j = cur.z * grp + jj;
            if (tid == 0) tma::wait_read();  // the previous P tile has left the staging buffer
            if (tid < C) {
                sg[tid] = gnext;
                lg[tid] = gnext * LOG2E - log2f(nk[tid]);
            }
            __syncthreads();
            // the next step's gates: the next value head of this item, or the first of the next item
            if (jj + 1 < grp)
                fetch_g(cur, j + 1);
            else if (nxt.y >= 0)
                fetch_g(nxt, nxt.z * grp);
            // P_rs = scale nq_r (Q K^T)_rs * 2^(G_r log2 e - LG_s) = scale nq_r nk_s e^(G_r - G_s) (Q K^T)_rs
            uint32_t w[16];
            if (zero_blk) {
#pragma unroll
                for (int u = 0; u < 16; ++u) w[u] = 0u;
            } else {
                const float gr2 = sg[r] * LOG2E;
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int s0 = half * 32 + 2 * u;
                    const float v0 = (s0 <= r && r < cur.y) ? exp2f(gr2 - lg[s0]) * x[2 * u] : 0.f;
                    const float v1 = (s0 + 1 <= r && r < cur.y) ? exp2f(gr2 - lg[s0 + 1]) * x[2 * u + 1] : 0.f;
                    w[u] = Elt<T>::pack(v0, v1);
                }
            }
            if (staged) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    umma::st_shared_v4(sb + S_PST + umma::off(r, half * 32 + c * 8, 0), w[4 * c], w[4 * c + 1],
                                       w[4 * c + 2], w[4 * c + 3]);
            } else if (r < cur.y) {
                T *dst = static_cast<T *>(p.P) + (((long long)cur.x + r) * Hv + j) * C + half * 32;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4 *>(dst + c * 8) = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
            }
            if (p.l2norm && r < cur.y) (half ? p.rk : p.rq)[((long long)cur.x + r) * Hv + j] = (half ? nk : nq)[r];
            if (staged) umma::fence_async_smem();
            __syncthreads();  // the gates of this step are read, the staged tile is complete
            if (staged && tid == 0) {
                tma::store3d(&p.tp, 0, j, cur.x, sb + S_PST);
                tma::commit_group();
            }
        }
        // TMEM, the norms and the gates are free for the next item
        umma::fence_before();
        __syncthreads();
        umma::fence_after();
        cur = nxt;
        stage = stage == NST - 1 ? 0 : stage + 1;
    }
    // after an error, let the loads and the MMA in flight finish before the block exits (bounded waits);
    // the P stores complete before shared memory goes away
    if (tid == 0) {
        for (int sx = 0; sx < NST; ++sx)
            if (iss[sx] > seen[sx]) umma::mbar_wait(full0 + 8u * (uint32_t)sx, (fph >> sx) & 1u, 4000000L);
        if (mma_out) umma::mbar_wait(mbar, mph, 4000000L);
        tma::wait_all();
    }
    umma::fence_before();
    __syncthreads();
    if (warp == 0) umma::dealloc(tmem, T_COLS);
}

template <typename T>
cudaError_t chunk_p_tc_t(const Args &a, const PpP &p, cudaStream_t s) {
    if (a.max_chunks == 0) return cudaSuccess;
    if ((long long)a.max_chunks * a.Hq >= (1ll << 31)) return cudaErrorInvalidValue;  // 32-bit item indices
    auto kern = chunk_p_tc_kernel<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S_BYTES);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const long items = (long)a.max_chunks * a.Hq;
    const unsigned grid = (unsigned)(items < 2L * sms ? items : 2L * sms);  // two persistent CTAs per SM
    return launch_plain(kern, dim3(grid), dim3(PT), S_BYTES, s, make_geo(a), p);
}

}  // namespace

cudaError_t launch_chunk_p_tc(const Args &a, const void *q, const void *k, const float *g_cs, void *P, float *rq,
                              float *rk, cudaStream_t s) {
    PpP p;
    const uint64_t tokens = (uint64_t)a.B * (uint64_t)a.T;
    const bool bf = a.bf16;
    if (!make_token_map(&p.tq, q, bf, a.K, a.Hq, tokens, 64) || !make_token_map(&p.tk, k, bf, a.K, a.Hq, tokens, 64) ||
        !make_tmap_3d(&p.tp, P, bf, C, a.Hv, tokens, C * 2, (uint64_t)a.Hv * C * 2, 64, 1, 64))
        return cudaErrorInvalidValue;
    p.g_cs = g_cs;
    p.P = P;
    p.rq = rq;
    p.rk = rk;
    p.l2norm = a.l2norm;
    p.scale = a.scale;
    p.nslots = (int)a.max_chunks;
    p.polls = a.wait_polls >= 0 ? (long)a.wait_polls : 200000000L;
    return a.bf16 ? chunk_p_tc_t<__nv_bfloat16>(a, p, s) : chunk_p_tc_t<__half>(a, p, s);
}

}  // namespace gdr
