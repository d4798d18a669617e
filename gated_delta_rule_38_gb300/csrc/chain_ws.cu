// Forward recurrence of the chunked gated delta rule, warp-specialised on the
// 5th-generation tensor cores (tcgen05 + TMEM, TMA tile loads).
//
// The columns of the state h = S^T [K x V] evolve independently, so one CTA of
// 512 threads owns one (sequence, value head, BV-wide slice of the value
// columns).  The slice of h lives in fp32 registers of eight "state" warps
// (TMEM lane = key row d) and, rounded, in shared memory as the B operand of
// the MMAs.  With G the chunk-local cumsum of g, Gl = G at the last valid row,
// rq / rk the inverse L2 norms of the q / k rows (1 without normalisation) and
// A = (I + strictly-lower(diag(beta)(K K^T o Gamma)))^-1 from wy_fwd, a chunk is
//
//   state-independent products, issued one chunk ahead so that they overlap
//   the previous chunk's recurrence:
//     [. ; Q] K^T                       -> Q K^T in TMEM lanes 64..127   (M=128, N=64, K=128)
//     K^T (A diag(beta e^G rk))^T       -> W^T                           (M=128, N=64, K=64)
//     [A diag(beta) ; 0] V              -> U in lanes 0..63, 0 above     (M=128, N=BV, K=64)
//     epilogues: -W^T and Q~^T = (diag(scale rq e^G) Q)^T into one MN-major operand;
//                K~ = diag(rk e^{Gl-G}) K in place; P = Q K^T o (scale rq_r rk_s e^{G_r-G_s}), s <= r
//   the recurrence, two dependent MMA rounds:
//     round A:  [-W ; Q~] h added to [U ; 0]  -> Delta (lanes 0..63), Q~ h (lanes 64..127)
//     round B:  X = K~^T Delta ;  [. ; P] Delta added to lanes 64..127 -> the output rows
//     epilogue: h <- e^{Gl} h + X
//
// This is the chunk form of S_t = e^{g_t} S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
// o_t = scale S_t q_t (FlashQLA skill page, "Core API"; gated delta rule chunk form with the
// WY/UT representation, PR #998 "[GDN] Add FlashQLA backend dispatch").
//
// Warp roles (one CTA per SM):
//   warp 0        lane 0 issues every MMA (single-thread issue, commits to mbarriers)
//   warp 1        lane 0 issues the TMA tile loads into a two-stage ring
//   warps 2, 3    TMEM lanes 64..127: the P epilogue and the output rows
//   warps 4..11   the state: TMEM lane 32*(w%4)+l, value columns of half (w-4)/4 of the slice
//   warps 12..15  per-chunk preparation: norms, gate factors, scaled copies of A, -W^T, Q~^T, K~
// Hand-offs go through mbarriers whose phases each complete once per chunk; every wait is
// bounded and gives up early once another role has raised the block's error flag.
#include <cuda_runtime.h>

#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tmap.h"
#include "umma.cuh"

namespace gdr {
namespace {

constexpr int WS_NT = 512;
constexpr long kWaitPolls = 40000000L;

// factor arrays (64 floats each), two sets (chunk parity)
enum { FG = 0, FRQ, FRK, FRQS, FCQ, FCK, FAKG, FAB, NF };

template <int BV>
struct Lay {
    // stage: [V b0 | Q b0 | A or V b1 | Q b1 | K b0 | K b1 (| A)], 8 KB blocks of 64 rows x 128 B
    static constexpr uint32_t ST_V = 0, ST_Q0 = 8192, ST_Q1 = 24576, ST_K0 = 32768;
    static constexpr uint32_t ST_A = BV == 128 ? 49152 : 16384;
    static constexpr uint32_t ST_BYTES = BV == 128 ? 57344 : 49152;
    static constexpr uint32_t WQ = 2 * ST_BYTES;  // MN-major [-W^T | Q~^T], 16 KB blocks of 128 d-rows
    static constexpr uint32_t AKG = WQ + 32768;   // [r][s] K-major
    static constexpr uint32_t PT0 = AKG + 8192;   // P of even chunks (its MMA reads AKG as rows 0..63)
    static constexpr uint32_t AB = PT0 + 8192;    // [r][s], followed by 8 KB of zeros
    static constexpr uint32_t Z = AB + 8192;
    static constexpr uint32_t DL = Z + 8192;       // Delta [64 s][BV]: BV/64 blocks of 8 KB
    static constexpr uint32_t PT1 = DL + BV * 128;  // P of odd chunks (rows 0..63 of its MMA: Delta)
    static constexpr uint32_t H = PT1 + 8192;       // h [128 d][BV]: BV/64 blocks of 16 KB
    static constexpr uint32_t F = H + BV * 256;
    static constexpr uint32_t BAR = F + 2 * NF * 256;
    // barriers
    static constexpr uint32_t B_FULL = BAR, B_EMPTY = BAR + 16, B_PREP = BAR + 32, B_EPIP = BAR + 40,
                              B_MP = BAR + 48, B_MA = BAR + 56, B_EPIA = BAR + 64, B_MB = BAR + 72,
                              B_EPIB = BAR + 80, B_MO = BAR + 88, B_OFREE = BAR + 104, B_DONE = BAR + 120;
    static constexpr uint32_t SLOT = BAR + 128, FLAG = SLOT + 4, USED = FLAG + 12;
    static constexpr uint32_t BYTES = USED + 1024;  // slack for aligning the base
    // TMEM columns
    static constexpr uint32_t T_D0 = 0, T_D1 = BV, T_X = 2 * BV, T_QK = 3 * BV, T_W = 3 * BV + 64;
};
static_assert(Lay<64>::BYTES <= 232448, "shared memory");

struct WsP {
    CUtensorMap tq, tk, tv, ta;  // [tokens][heads][cols] maps, boxes 64 x 1 x 64
    const float *g_cs, *h0;
    const void *beta;
    void *o;
    float *fin;
    void *h;       // optional: state before every chunk, [rows,Hv,K,V] (or [..,V,K] with h_vfirst)
    void *delta;   // optional: Delta of every chunk, [rows,Hv,64,V]
    const float *seg_start;  // optional start states, transposed [N,Hv,V,K] fp32 (replaces h0)
    bool gate_f32, l2norm, v_first, h_vfirst;
    float scale;
};

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

// Wait for the phase of `bar` with the given parity.  Gives up when the block's flag is raised by
// another role, or after a bound (then it latches GDR_ERR_TIMEOUT and raises the flag itself).
__device__ __noinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int *flag, unsigned *err) {
    for (long it = 0; it < kWaitPolls; ++it) {
        if (mbar_try(bar, parity)) return true;
        if ((it & 127) == 127 && *flag) return false;
    }
    raise_error(err, GDR_ERR_TIMEOUT);
    *flag = 1;
    return false;
}

// Warp-uniform wait: lane 0 polls, the warp agrees on the outcome and synchronises its memory view.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *flag, unsigned *err, int lane) {
    int ok = 0;
    if (lane == 0) ok = wait_phase(bar, parity, flag, err) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

// Barrier `id` over `nthreads` threads that also ANDs a predicate across them.
__device__ __forceinline__ bool group_and(bool v, int id, int nthreads) {
    uint32_t r;
    asm volatile(
        "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.and.pred q, %2, %3, p;\nselp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

template <typename T> struct IsBf16 { static constexpr bool value = false; };
template <> struct IsBf16<__nv_bfloat16> { static constexpr bool value = true; };

__device__ __forceinline__ void st_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    umma::st_shared_v4(addr, a, b, c, d);
}

// 16 fp32 values -> 8 packed pairs -> two 16-byte stores at columns col0.. of a swizzled row.
template <typename T>
__device__ __forceinline__ void store_row16(uint32_t blk, int row, int col0, const float *x) {
#pragma unroll
    for (int c = 0; c < 2; ++c)
        st_v4(blk + umma::off(row, col0 + c * 8, 0), Elt<T>::pack(x[c * 8], x[c * 8 + 1]),
              Elt<T>::pack(x[c * 8 + 2], x[c * 8 + 3]), Elt<T>::pack(x[c * 8 + 4], x[c * 8 + 5]),
              Elt<T>::pack(x[c * 8 + 6], x[c * 8 + 7]));
}

template <typename T>
__device__ __forceinline__ uint16_t to_bits(float x) {
    const T h = Elt<T>::from_f(x);
    return *reinterpret_cast<const uint16_t *>(&h);
}

template <typename T, int BV, bool WRITE_O>
__global__ void __launch_bounds__(WS_NT, 1) chain_ws_kernel(Geo geo, const __grid_constant__ WsP p) {
    using L = Lay<BV>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const int vh = blockIdx.x, j = blockIdx.y, n = blockIdx.z;
    const int v0 = vh * BV;
    const int Hv = geo.Hv, Hq = geo.Hq, hq = j / (Hv / Hq);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr bool bf16 = IsBf16<T>::value;
    long long tok0;
    int len, row0;
    geo.seq(n, tok0, len, row0);
    const int nc = (len + C - 1) / C;
    volatile int *flag = reinterpret_cast<volatile int *>(smem + L::FLAG);
    float *F = reinterpret_cast<float *>(smem + L::F);
    auto fa = [&](int par, int which) -> float * { return F + (par * NF + which) * 64; };

    if (tid == 0) {
        umma::mbar_init(sb + L::B_FULL, 1);
        umma::mbar_init(sb + L::B_FULL + 8, 1);
        umma::mbar_init(sb + L::B_EMPTY, 1);
        umma::mbar_init(sb + L::B_EMPTY + 8, 1);
        umma::mbar_init(sb + L::B_PREP, 4);
        umma::mbar_init(sb + L::B_EPIP, WRITE_O ? 6 : 4);
        umma::mbar_init(sb + L::B_MP, 2);  // the commit, and the issuing thread's own arrival
        umma::mbar_init(sb + L::B_MA, 1);
        umma::mbar_init(sb + L::B_EPIA, 4);
        umma::mbar_init(sb + L::B_MB, 1);
        umma::mbar_init(sb + L::B_EPIB, 8);
        umma::mbar_init(sb + L::B_MO, 1);
        umma::mbar_init(sb + L::B_MO + 8, 1);
        umma::mbar_init(sb + L::B_OFREE, 2);
        umma::mbar_init(sb + L::B_OFREE + 8, 2);
        umma::mbar_init(sb + L::B_DONE, 1);
        umma::fence_mbar_init();
        *flag = 0;
    }
    // zero block below A diag(beta) (rows 64..127 of the U product)
    for (int i = tid; i < 8192 / 16; i += WS_NT) st_v4(sb + L::Z + i * 16, 0u, 0u, 0u, 0u);
    umma::fence_async_smem();
    if (warp == 0) umma::alloc(sb + L::SLOT, 512);
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::SLOT);

    if (warp == 1) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued[2] = {0, 0};
            for (int lc = 0; lc < nc && !*flag; ++lc) {
                const int s = lc & 1;
                if (lc >= 2 && !wait_phase(sb + L::B_EMPTY + 8 * s, ((lc >> 1) - 1) & 1, flag, geo.err)) break;
                const uint32_t st = sb + s * L::ST_BYTES, full = sb + L::B_FULL + 8 * s;
                const int t = (int)(tok0 + (long long)lc * C);
                tma::expect_tx(full, (WRITE_O ? 16384u : 0u) + 16384u + (uint32_t)BV * 128u + 8192u);
                if (WRITE_O) {
                    tma::load3d(st + L::ST_Q0, &p.tq, 0, hq, t, full);
                    tma::load3d(st + L::ST_Q1, &p.tq, 64, hq, t, full);
                }
                tma::load3d(st + L::ST_K0, &p.tk, 0, hq, t, full);
                tma::load3d(st + L::ST_K0 + 8192, &p.tk, 64, hq, t, full);
                tma::load3d(st + L::ST_V, &p.tv, v0, j, t, full);
                if (BV == 128) tma::load3d(st + L::ST_V + 16384, &p.tv, v0 + 64, j, t, full);
                tma::load3d(st + L::ST_A, &p.ta, 0, j, t, full);
                ++issued[s];
            }
            // let every load in flight land before the block can exit (bounded)
            for (int s = 0; s < 2; ++s)
                if (issued[s] > 0) umma::mbar_wait(sb + L::B_FULL + 8 * s, (issued[s] - 1) & 1, 4000000L);
        }
    } else if (warp == 0) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint32_t id_qk = umma::idesc(128, 64, bf16, false, false);
            const uint32_t id_w = umma::idesc(128, 64, bf16, true, false);
            const uint32_t id_u = umma::idesc(128, BV, bf16, false, true);
            const uint32_t id_mn = umma::idesc(128, BV, bf16, true, true);
            const uint32_t id_o = umma::idesc(128, BV, bf16, false, true);
            const uint64_t dAKG = umma::desc(sb + L::AKG, 16, 1024), dAB = umma::desc(sb + L::AB, 16, 1024);
            const uint64_t dWQ = umma::desc(sb + L::WQ, 16384, 1024), dH = umma::desc(sb + L::H, 16384, 1024);
            const uint64_t dDL = umma::desc(sb + L::DL, 8192, 1024);
            const uint64_t dP0 = umma::desc(sb + L::PT0 - 8192, 16, 1024), dP1 = umma::desc(sb + L::PT1 - 8192, 16, 1024);
            auto issue_p = [&](int lc) {
                const int s = lc & 1;
                const uint32_t st = sb + s * L::ST_BYTES;
                if (WRITE_O) {
                    const uint64_t aq = umma::desc(st, 16, 1024), bk = umma::desc(st + L::ST_K0, 16, 1024);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        umma::mma(tmem + L::T_QK, aq + ((((ks >> 2) * 16384) + (ks & 3) * 32) >> 4),
                                  bk + ((((ks >> 2) * 8192) + (ks & 3) * 32) >> 4), id_qk, ks > 0);
                }
                const uint64_t akmn = umma::desc(st + L::ST_K0, 8192, 1024), bv = umma::desc(st + L::ST_V, 16384, 1024);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    umma::mma(tmem + L::T_W, akmn + ks * 128, dAKG + ks * 2, id_w, ks > 0);
                    umma::mma(tmem + (s ? L::T_D1 : L::T_D0), dAB + ks * 2, bv + ks * 128, id_u, ks > 0);
                }
                umma::commit(sb + L::B_MP);
                mbar_arrive(sb + L::B_MP);
            };
            bool ok = true;
            if (nc > 0) {
                ok = wait_phase(sb + L::B_PREP, 0, flag, geo.err) && wait_phase(sb + L::B_FULL, 0, flag, geo.err);
                umma::fence_after();
                if (ok) issue_p(0);
            }
            for (int lc = 0; lc < nc && ok; ++lc) {
                const int b = lc & 1;
                const uint32_t st = sb + b * L::ST_BYTES;
                const uint32_t tD = b ? L::T_D1 : L::T_D0;
                // round A: needs this chunk's -W^T / Q~^T / K~ / P and the state tile
                if (!(ok = wait_phase(sb + L::B_EPIP, lc & 1, flag, geo.err) &&
                           wait_phase(sb + L::B_EPIB, lc & 1, flag, geo.err)))
                    break;
                umma::fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) umma::mma(tmem + tD, dWQ + ks * 128, dH + ks * 128, id_mn, true);
                umma::commit(sb + L::B_MA);
                // the next chunk's state-independent products run while round A's epilogue works
                if (lc + 1 < nc) {
                    const int b1 = (lc + 1) & 1;
                    if (!(ok = wait_phase(sb + L::B_PREP, (lc + 1) & 1, flag, geo.err) &&
                               wait_phase(sb + L::B_FULL + 8 * b1, ((lc + 1) >> 1) & 1, flag, geo.err) &&
                               (!WRITE_O || lc < 1 || wait_phase(sb + L::B_OFREE + 8 * b1, ((lc - 1) >> 1) & 1, flag, geo.err))))
                        break;
                    umma::fence_after();
                    issue_p(lc + 1);
                }
                // round B: needs Delta
                if (!(ok = wait_phase(sb + L::B_EPIA, lc & 1, flag, geo.err))) break;
                umma::fence_after();
                const uint64_t akt = umma::desc(st + L::ST_K0, 8192, 1024);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    umma::mma(tmem + L::T_X, akt + ks * 128, dDL + ks * 128, id_mn, ks > 0);
                    if (WRITE_O) umma::mma(tmem + tD, (b ? dP1 : dP0) + ks * 2, dDL + ks * 128, id_o, true);
                }
                umma::commit(sb + L::B_MB);
                umma::commit(sb + L::B_EMPTY + 8 * b);
                umma::commit(sb + L::B_MO + 8 * b);
            }
            // every MMA issued so far completes before TMEM is released
            umma::commit(sb + L::B_DONE);
            umma::mbar_wait(sb + L::B_DONE, 0, 4000000L);
        }
    } else if (warp >= 12) {
        // ------------------------------------------------------------ preparation (128 threads)
        const int at = tid - 384;
        const int lb = (warp & 3) * 32;  // == at & ~31
        float greg = 0.f, breg = 0.f;
        auto fetch = [&](int lc) {
            const int valid = min(C, len - lc * C);
            const int r = at & 63;
            if (r < valid) {
                const long long ti = (tok0 + (long long)lc * C + r) * Hv + j;
                if (at < 64)
                    greg = p.g_cs[ti];
                else
                    breg = load_gate<T>(p.beta, ti, p.gate_f32);
            } else {
                greg = 0.f;
                breg = 0.f;
            }
        };
        if (nc > 0) fetch(0);
        for (int lc = 0; lc < nc; ++lc) {
            const int b = lc & 1, s = lc & 1;
            const uint32_t st = sb + s * L::ST_BYTES;
            const int valid = min(C, len - lc * C);
            if (at < 64)
                fa(b, FG)[at] = greg;
            else
                fa(b, FAB)[at - 64] = breg;  // raw beta for now
            if (lc + 1 < nc) fetch(lc + 1);
            if (!group_and(warp_wait(sb + L::B_FULL + 8 * s, (lc >> 1) & 1, flag, geo.err, lane), 1, 128)) break;
            // inverse norms of the q rows (threads 0..63) and k rows (64..127)
            if (p.l2norm && (WRITE_O || at >= 64)) {
                const int r = at & 63;
                const uint32_t b0 = st + (at < 64 ? L::ST_Q0 : L::ST_K0);
                const uint32_t b1 = st + (at < 64 ? L::ST_Q1 : L::ST_K0 + 8192);
                float ss = 0.f;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const uint4 u = umma::ld_shared_v4((c < 8 ? b0 : b1) + umma::off(r, (c & 7) * 8, 0));
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 x = Elt<T>::unpack(w[e]);
                        ss = fmaf(x.x, x.x, fmaf(x.y, x.y, ss));
                    }
                }
                fa(b, at < 64 ? FRQ : FRK)[r] = 1.0f / sqrtf(ss + L2_EPS);
            }
            asm volatile("bar.sync 1, 128;\n" ::: "memory");
            if (at < 64) {
                const int r = at;
                const bool ok = r < valid;
                const float gr = fa(b, FG)[r], Gl = fa(b, FG)[valid - 1];
                const float rq = (p.l2norm && WRITE_O) ? fa(b, FRQ)[r] : 1.f;
                const float rk = p.l2norm ? fa(b, FRK)[r] : 1.f;
                const float be = fa(b, FAB)[r];
                const float eg = __expf(gr);
                fa(b, FRQS)[r] = ok ? p.scale * rq : 0.f;
                fa(b, FRK)[r] = ok ? rk : 0.f;
                fa(b, FCQ)[r] = ok ? p.scale * rq * eg : 0.f;
                fa(b, FCK)[r] = ok ? rk * __expf(Gl - gr) : 0.f;
                fa(b, FAKG)[r] = ok ? be * eg * rk : 0.f;
                fa(b, FAB)[r] = ok ? be : 0.f;
            }
            asm volatile("bar.sync 1, 128;\n" ::: "memory");
            // A diag(beta e^G rk) and A diag(beta): thread -> row at/2, 32 columns; rows past the end are zero
            {
                const int r = at >> 1, c0 = (at & 1) * 32;
                const float *fk = fa(b, FAKG), *fb = fa(b, FAB);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int col = c0 + c * 8;
                    const uint32_t o = umma::off(r, col, 0);
                    const uint4 u = umma::ld_shared_v4(st + L::ST_A + o);
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
                    uint32_t wk[4], wb[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 x = Elt<T>::unpack(w[e]);
                        const bool ok = r < valid;
                        wk[e] = Elt<T>::pack(ok ? x.x * fk[col + 2 * e] : 0.f, ok ? x.y * fk[col + 2 * e + 1] : 0.f);
                        wb[e] = Elt<T>::pack(ok ? x.x * fb[col + 2 * e] : 0.f, ok ? x.y * fb[col + 2 * e + 1] : 0.f);
                    }
                    st_v4(sb + L::AKG + o, wk[0], wk[1], wk[2], wk[3]);
                    st_v4(sb + L::AB + o, wb[0], wb[1], wb[2], wb[3]);
                }
            }
            umma::fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(sb + L::B_PREP);
            // ---- after the state-independent products of this chunk
            if (!group_and(warp_wait(sb + L::B_MP, lc & 1, flag, geo.err, lane), 1, 128)) break;
            umma::fence_after();
            {
                // -W^T row d = at: 64 token columns into the MN-major block 0 of WQ
#pragma unroll
                for (int c = 0; c < 64; c += 16) {
                    float x[16];
                    umma::ld16(umma::taddr(tmem, lb, L::T_W + c), x);
                    umma::ld_wait();
#pragma unroll
                    for (int u = 0; u < 16; ++u) x[u] = -x[u];
                    store_row16<T>(sb + L::WQ, at, c, x);
                }
            }
            umma::fence_before();
            if (WRITE_O) {
                // Q~^T: thread -> q row r = at & 63, key half at >> 6; element (d, r) of block 1 of WQ
                const int r = at & 63, dh = at >> 6;
                const float cq = fa(b, FCQ)[r];
                const uint32_t src = st + (dh ? L::ST_Q1 : L::ST_Q0), dst = sb + L::WQ + 16384;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 u = umma::ld_shared_v4(src + umma::off(r, c * 8, 0));
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 x = Elt<T>::unpack(w[e]);
                        const int d = dh * 64 + c * 8 + 2 * e;
                        const uint16_t lo = to_bits<T>(x.x * cq), hi = to_bits<T>(x.y * cq);
                        asm volatile("st.shared.u16 [%0], %1;\n" ::"r"(dst + umma::off(d, r, 0)), "h"(lo));
                        asm volatile("st.shared.u16 [%0], %1;\n" ::"r"(dst + umma::off(d + 1, r, 0)), "h"(hi));
                    }
                }
            }
            {
                // K~ in place: thread -> k row s = at & 63, key half at >> 6
                const int s2 = at & 63, dh = at >> 6;
                const float ck = fa(b, FCK)[s2];
                const uint32_t blk = st + L::ST_K0 + dh * 8192;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t a = blk + umma::off(s2, c * 8, 0);
                    const uint4 u = umma::ld_shared_v4(a);
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
                    uint32_t o4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 x = Elt<T>::unpack(w[e]);
                        o4[e] = Elt<T>::pack(x.x * ck, x.y * ck);
                    }
                    st_v4(a, o4[0], o4[1], o4[2], o4[3]);
                }
            }
            umma::fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(sb + L::B_EPIP);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ state (256 threads)
        const int sw = warp - 4, q4 = warp & 3, cg = sw >> 2;
        const int d = q4 * 32 + lane;  // TMEM lane: key row of h, token row of Delta
        constexpr int HW = BV / 2;     // value columns per thread
        const int cb0 = cg * HW;
        const long long st_base = ((long long)n * Hv + j) * DK * DV;
        float hS[HW];
#pragma unroll
        for (int i = 0; i < HW; ++i) {
            const int e = v0 + cb0 + i;
            if (p.seg_start)
                hS[i] = p.seg_start[st_base + (long long)e * DK + d];
            else if (p.h0)
                hS[i] = p.h0[st_base + (p.v_first ? (long long)e * DK + d : (long long)d * DV + e)];
            else
                hS[i] = 0.f;
        }
        auto write_h = [&]() {
#pragma unroll
            for (int i = 0; i < HW; i += 16) {
                const int col = cb0 + i;
                store_row16<T>(sb + L::H + (col >> 6) * 16384, d, col & 63, hS + i);
            }
            umma::fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(sb + L::B_EPIB);
        };
        write_h();
        float glo = 0.f;
        auto fetch_gl = [&](int lc) {
            const int valid = min(C, len - lc * C);
            glo = p.g_cs[(tok0 + (long long)lc * C + valid - 1) * Hv + j];
        };
        if (nc > 0) fetch_gl(0);
        for (int lc = 0; lc < nc; ++lc) {
            const int b = lc & 1;
            const uint32_t tD = b ? L::T_D1 : L::T_D0;
            const float egl = __expf(glo);
            if (lc + 1 < nc) fetch_gl(lc + 1);
            if (p.h) {
                // the state before this chunk
                T *hb = static_cast<T *>(p.h) + ((long long)(row0 + lc) * Hv + j) * DK * DV;
                if (p.h_vfirst) {
#pragma unroll
                    for (int i = 0; i < HW; ++i) hb[(long long)(v0 + cb0 + i) * DK + d] = Elt<T>::from_f(hS[i]);
                } else {
                    T *hr = hb + (long long)d * DV + v0 + cb0;
#pragma unroll
                    for (int i = 0; i < HW; i += 8)
                        *reinterpret_cast<uint4 *>(hr + i) =
                            make_uint4(Elt<T>::pack(hS[i], hS[i + 1]), Elt<T>::pack(hS[i + 2], hS[i + 3]),
                                       Elt<T>::pack(hS[i + 4], hS[i + 5]), Elt<T>::pack(hS[i + 6], hS[i + 7]));
                }
            }
            if (q4 < 2) {
                // Delta rows (lanes 0..63) -> the B operand of round B
                if (!warp_wait(sb + L::B_MA, lc & 1, flag, geo.err, lane)) break;
                umma::fence_after();
#pragma unroll
                for (int i = 0; i < HW; i += 16) {
                    float x[16];
                    umma::ld16(umma::taddr(tmem, q4 * 32, tD + cb0 + i), x);
                    umma::ld_wait();
                    const int col = cb0 + i;
                    store_row16<T>(sb + L::DL + (col >> 6) * 8192, d, col & 63, x);
                    if (p.delta) {
                        T *dr = static_cast<T *>(p.delta) + (((long long)(row0 + lc) * Hv + j) * C + d) * DV + v0 + col;
                        uint4 w0, w1;
                        w0 = make_uint4(Elt<T>::pack(x[0], x[1]), Elt<T>::pack(x[2], x[3]), Elt<T>::pack(x[4], x[5]),
                                        Elt<T>::pack(x[6], x[7]));
                        w1 = make_uint4(Elt<T>::pack(x[8], x[9]), Elt<T>::pack(x[10], x[11]),
                                        Elt<T>::pack(x[12], x[13]), Elt<T>::pack(x[14], x[15]));
                        *reinterpret_cast<uint4 *>(dr) = w0;
                        *reinterpret_cast<uint4 *>(dr + 8) = w1;
                    }
                }
                umma::fence_before();
                umma::fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(sb + L::B_EPIA);
            }
            if (!warp_wait(sb + L::B_MB, lc & 1, flag, geo.err, lane)) break;
            umma::fence_after();
#pragma unroll
            for (int i = 0; i < HW; i += 16) {
                float x[16];
                umma::ld16(umma::taddr(tmem, q4 * 32, L::T_X + cb0 + i), x);
                umma::ld_wait();
#pragma unroll
                for (int u = 0; u < 16; ++u) hS[i + u] = fmaf(egl, hS[i + u], x[u]);
            }
            umma::fence_before();
            write_h();
        }
        if (!*flag && p.fin) {
#pragma unroll
            for (int i = 0; i < HW; ++i) {
                const int e = v0 + cb0 + i;
                p.fin[st_base + (p.v_first ? (long long)e * DK + d : (long long)d * DV + e)] = hS[i];
            }
        }
    } else if (WRITE_O) {
        // ------------------------------------------------------------ P and output rows (warps 2, 3)
        const int r = tid - 64;  // token row; TMEM lane 64 + r
        const int lb = 32 * (warp & 3);
        for (int lc = 0; lc < nc; ++lc) {
            const int b = lc & 1;
            const int valid = min(C, len - lc * C);
            if (!warp_wait(sb + L::B_MP, lc & 1, flag, geo.err, lane)) break;
            umma::fence_after();
            {
                const float *fg = fa(b, FG), *frk = fa(b, FRK);
                const float gr = fg[r], rr = fa(b, FRQS)[r];
                const uint32_t dst = sb + (b ? L::PT1 : L::PT0);
#pragma unroll
                for (int c = 0; c < 64; c += 16) {
                    float x[16];
                    umma::ld16(umma::taddr(tmem, lb, L::T_QK + c), x);
                    umma::ld_wait();
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const int s2 = c + u;
                        x[u] = (s2 <= r && r < valid) ? x[u] * rr * frk[s2] * __expf(gr - fg[s2]) : 0.f;
                    }
                    store_row16<T>(dst, r, c, x);
                }
            }
            umma::fence_before();
            umma::fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(sb + L::B_EPIP);
            if (!warp_wait(sb + L::B_MO + 8 * b, (lc >> 1) & 1, flag, geo.err, lane)) break;
            umma::fence_after();
            {
                const uint32_t tD = b ? L::T_D1 : L::T_D0;
                T *orow = static_cast<T *>(p.o) + ((tok0 + (long long)lc * C + r) * Hv + j) * DV + v0;
#pragma unroll
                for (int c = 0; c < BV; c += 16) {
                    float x[16];
                    umma::ld16(umma::taddr(tmem, lb, tD + c), x);
                    umma::ld_wait();
                    if (r < valid) {
                        *reinterpret_cast<uint4 *>(orow + c) =
                            make_uint4(Elt<T>::pack(x[0], x[1]), Elt<T>::pack(x[2], x[3]), Elt<T>::pack(x[4], x[5]),
                                       Elt<T>::pack(x[6], x[7]));
                        *reinterpret_cast<uint4 *>(orow + c + 8) =
                            make_uint4(Elt<T>::pack(x[8], x[9]), Elt<T>::pack(x[10], x[11]),
                                       Elt<T>::pack(x[12], x[13]), Elt<T>::pack(x[14], x[15]));
                    }
                }
            }
            umma::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(sb + L::B_OFREE + 8 * b);
        }
    }

    umma::fence_before();
    __syncthreads();
    if (warp == 0) umma::dealloc(tmem, 512);
}

bool ws_map(CUtensorMap *m, const void *base, const Args &a, int heads, int cols) {
    const uint64_t tokens = (uint64_t)a.B * (uint64_t)a.T;
    return make_tmap_3d(m, base, a.bf16, (uint64_t)cols, (uint64_t)heads, tokens, (uint64_t)cols * 2,
                        (uint64_t)heads * cols * 2, 64, 1, 64);
}

template <typename T, int BV, bool WRITE_O>
cudaError_t chain_ws_t(const Args &a, const WsP &p, cudaStream_t s) {
    auto kern = chain_ws_kernel<T, BV, WRITE_O>;
    const uint32_t bytes = Lay<BV>::BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    kern<<<dim3(DV / BV, a.Hv, a.N), WS_NT, bytes, s>>>(make_geo(a), p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chain_ws(const Args &a, const void *q, const void *k, const void *v, const float *g_cs,
                            const void *beta, const void *A, const float *h0, const float *seg_start, void *o,
                            float *final_state, void *h, bool h_vfirst, void *delta, cudaStream_t s) {
    WsP p;
    if (!ws_map(&p.tq, q, a, a.Hq, DK) || !ws_map(&p.tk, k, a, a.Hq, DK) || !ws_map(&p.tv, v, a, a.Hv, DV) ||
        !ws_map(&p.ta, A, a, a.Hv, C))
        return cudaErrorInvalidValue;
    p.g_cs = g_cs;
    p.h0 = h0;
    p.beta = beta;
    p.o = o;
    p.fin = final_state;
    p.h = h;
    p.delta = delta;
    p.seg_start = seg_start;
    p.gate_f32 = a.gate_f32;
    p.l2norm = a.l2norm;
    p.v_first = a.v_first;
    p.h_vfirst = h_vfirst;
    p.scale = a.scale;
    if (o)
        return a.bf16 ? chain_ws_t<__nv_bfloat16, 64, true>(a, p, s) : chain_ws_t<__half, 64, true>(a, p, s);
    return a.bf16 ? chain_ws_t<__nv_bfloat16, 64, false>(a, p, s) : chain_ws_t<__half, 64, false>(a, p, s);
}

}  // namespace gdr
