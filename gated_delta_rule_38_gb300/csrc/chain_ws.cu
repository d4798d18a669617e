// Forward recurrence of the chunked gated delta rule, warp-specialised on the
// 5th-generation tensor cores (tcgen05 + TMEM, TMA tile loads).
//
// The columns of the state h = S^T [K x V] evolve independently, so one CTA of
// 512 threads owns one (sequence, value head, BV-wide slice of the value
// columns).  The slice of h lives in fp32 registers of eight "state" warps
// (TMEM lane = key row d) and, rounded, in shared memory as the B operand of
// the MMAs.  With G the chunk-local cumsum of g, Gl = G at the last valid row,
// rq / rk the inverse L2 norms of the q / k rows (1 without normalisation),
// A = (I + strictly-lower(diag(beta)(K K^T o Gamma)))^-1 and the decayed causal
// block P = scale (q^ k^T o Gamma) from wy_fwd, a chunk is
//
//   state-independent products, issued while the previous chunk's recurrence runs:
//     [0 ; A diag(beta e^G rk)] K   -> W in TMEM lanes 64..127                (M=128, N=128, K=64)
//     [A diag(beta) ; 0] V          -> U in lanes 0..63, 0 in 64..127         (M=128, N=BV,  K=64)
//     the -W epilogue fills the rows above Q in the stage
//   the recurrence, two dependent MMA rounds:
//     round A:  [-W ; Q] h added to [U ; 0]   -> Delta = U - W h (lanes 0..63), Q h (64..127)
//     round B:  X = K^T (diag(rk e^{Gl-G}) Delta) ;  [. ; P] Delta -> its own columns (lanes 64..127)
//     epilogues: h <- e^{Gl} h + X ; output rows o = diag(scale rq e^G) Q h + P Delta
//
// This is the chunk form of S_t = e^{g_t} S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
// o_t = scale S_t q_t (FlashQLA skill page, "Core API"; gated delta rule chunk form with the
// WY/UT representation, PR #998 "[GDN] Add FlashQLA backend dispatch").
//
// Warp roles (one CTA per SM):
//   warp 0            the MMA warp: the whole warp runs the loop and polls, lane 0 issues every MMA but
//                     round B's X (the next chunk's products go in small groups around round B so that
//                     round B never waits behind them)
//   warp 1            the TMA warp, likewise: tile loads into a two-stage ring, and an L2 prefetch of the
//                     next chunk's boxes
//   warps 2,3         TMEM lanes 64..127: the -W epilogue and the output rows
//   warps 4..11       the state: TMEM lane 32*(w%4)+l, value columns of half (w-4)/4 of the slice;
//                     warps 4,5,8,9 also move Delta (lanes 0..63) into shared memory, and warp 4 then issues
//                     round B's X product
//   warps 12..15      per-chunk preparation (one warp per scheduler): gate factors, scaled copies of A
// Hand-offs go through mbarriers whose phases each complete once per chunk (every lane of a waiting warp
// polls); every wait is bounded and gives up early once another role has raised the block's error flag.
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

// factor arrays (64 floats each), four sets (chunk index mod 4)
enum { FG = 0, FRQ, FRK, FB, FCQ, FCK, FAKG, FAB, NF };

template <int BV, bool WRITE_O = true>
struct Lay {
    // stage, 8 KB blocks of 64 rows x 128 B:
    //   with the output: [-W b0 | Q b0 | -W b1 | Q b1 | K b0 | K b1 | V | A | P]
    //   without it:      [-W b0 | K b0 | -W b1 | K b1 | V | A]      (K doubles as the idle rows of round A)
    // ([-W; Q] (or [-W; K]) is one K-major 128-row operand per key half, [A; P] one 128-row operand)
    static constexpr uint32_t ST_W0 = 0, ST_Q0 = 8192, ST_W1 = 16384, ST_Q1 = 24576;
    static constexpr uint32_t ST_K0 = WRITE_O ? 32768 : 8192, ST_K1 = WRITE_O ? 40960 : 24576;
    static constexpr uint32_t LBO_K = ST_K1 - ST_K0;
    static constexpr uint32_t ST_V = WRITE_O ? 49152 : 32768, ST_A = ST_V + BV * 128, ST_P = ST_A + 8192;
    static constexpr uint32_t ST_BYTES = WRITE_O ? ST_P + 8192 : ST_A + 8192;
    static constexpr uint32_t AB = 2 * ST_BYTES;  // [A diag(beta) ; 0] and [0 ; A diag(beta e^G rk)]
    static constexpr uint32_t Z = AB + 8192;
    static constexpr uint32_t AKG = Z + 8192;
    static constexpr uint32_t DT = AKG + 8192;                    // diag(rk e^{Gl-G}) Delta [64 s][BV]
    static constexpr uint32_t DL = DT + BV * 128;                 // Delta (output product; stored Delta)
    static constexpr uint32_t H = DL + BV * 128;                  // h [128 d][BV]: BV/64 blocks of 16 KB
    static constexpr uint32_t F = H + BV * 256;                   // factor sets (4, by chunk index mod 4)
    static constexpr uint32_t OST = F + 4 * NF * 256;             // output rows of a full chunk [64][BV]
    static constexpr uint32_t BAR = OST + (WRITE_O ? BV * 128 : 0);
    // barriers
    static constexpr uint32_t B_FULL = BAR, B_EMPTY = BAR + 16, B_PREP = BAR + 32,
                              B_MPW = BAR + 48, B_MA = BAR + 56, B_EPIA = BAR + 64, B_MB = BAR + 72,
                              B_EPIB = BAR + 80, B_MO = BAR + 88, B_OFREE = BAR + 104, B_DONE = BAR + 120,
                              B_MPU = BAR + 128;
    // the stage is loaded and released in two groups: "early" (q, v, A: done after round A) and "late"
    // (k, P: done after round B); B_FULL / B_EMPTY belong to the early group
    static constexpr uint32_t B_FULLL = BAR + 136, B_EMPTYL = BAR + 152;
    static constexpr uint32_t SLOT = BAR + 168, FLAG = SLOT + 4, USED = FLAG + 12;
    static constexpr uint32_t BYTES = USED + 1024;  // slack for aligning the base
    // TMEM columns
    static constexpr uint32_t T_W = 0, T_D0 = 128, T_D1 = 128 + BV, T_X = 128 + 2 * BV;
    // P Delta of the output rows, by chunk parity (lanes 64..127; with the output only)
    static constexpr uint32_t T_PD0 = 128 + 3 * BV, T_PD1 = 128 + 4 * BV;
};
static_assert(Lay<64>::BYTES <= 232448 && Lay<128, false>::BYTES <= 232448, "shared memory");
static_assert(Lay<128, false>::T_X + 128 <= 512 && Lay<64>::T_PD1 + 64 <= 512, "tensor memory");

struct WsP {
    CUtensorMap tq, tk, tv, tp, ta;  // [tokens][heads][cols] maps, boxes 64 x 1 x 64
    const float *g_cs, *h0, *rq, *rk;  // rq, rk: inverse q/k norms [tokens,Hv] (l2norm only)
    const void *beta;
    void *o;
    float *fin;
    void *h;       // optional: state before every chunk, [rows,Hv,K,V] (or [..,V,K] with h_vfirst)
    void *delta;   // optional: Delta of every chunk, [rows,Hv,64,V]
    const float *seg_start;  // optional start states, transposed [N,Hv,nseg,V,K] fp32 (replaces h0)
    int nseg;                // segments per sequence (the intra-GPU split; 1 = none): grid z = N x nseg
    // the split's segment-affine pass (BV = 128, no output): block x = kind, 0 = zero start with the values,
    // 1 = identity start with zero values (U = 0); every segment's end state, transposed, into
    // seg_end[kind] [N,Hv,nseg,V,K] fp32
    bool affine;
    float *seg_end[2];
    bool gate_f32, l2norm, v_first, h_vfirst;
    float scale;
    // with all 128 value columns in one CTA and the [K,V] layout, h and Delta leave by TMA store from the
    // bf16 tiles in shared memory: each state warp stores its own 32-row x 64-column box
    bool tma_h, tma_delta;
    CUtensorMap th, tdl;  // h [rows*Hv][128][128], Delta [rows*Hv][64][128]; boxes 64 x 32 x 1
    CUtensorMap to;       // o [tokens][Hv][V], boxes 64 x 1 x 32 (full chunks' output rows)
};

// One non-blocking test (the MMA thread polls several barriers in turn).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

// Wait for the phase of `bar` with the given parity.  Gives up when the block's flag is raised by
// another role, or after a bound (then it latches GDR_ERR_TIMEOUT and raises the flag itself).  It spins
// on a non-suspending test: a thread suspended in try_wait for long was seen to resume several hundred
// cycles after the phase completed, on the chain's critical path (only one lane of a waiting warp polls).
__device__ __noinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int *flag, unsigned *err) {
    for (long it = 0; it < kWaitPolls; ++it) {
        if (mbar_test(bar, parity)) return true;
        if ((it & 127) == 127 && *flag) return false;
    }
    raise_error(err, GDR_ERR_TIMEOUT);
    *flag = 1;
    return false;
}

// Warp-uniform wait: every lane polls and the warp agrees on the outcome.  (Lane 0 polling alone while
// the other lanes waited in a shuffle passed the phases markedly later: the forward chain ran 19 us slower.)
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *flag, unsigned *err, int lane) {
    (void)lane;
    return __all_sync(0xffffffffu, wait_phase(bar, parity, flag, err));
}

// Named-barrier arrival without waiting, and arrival with waiting, over `nthreads` threads.
__device__ __forceinline__ void bar_arrive(int id, int nthreads) {
    asm volatile("bar.arrive %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

// TMA stores of the state warps' tiles.  Each state warp holds 32 rows (its TMEM lane quadrant q4) of
// HW = BV/2 columns; a stored box is 32 rows x 64 columns.  With BV = 128 a warp owns its box; with BV = 64
// warps 4+q4 (cg 0, which issues the store) and 8+q4 (cg 1) share one, and two hardware barriers per pair
// order the hand-offs: barrier 4+q4 "the box stored from this tile last time has been read" (issuer
// arrives, partner waits), barrier 8+q4 "the partner's rows are written" (partner arrives, issuer waits).
// Both warps of a pair pass the same sequence of these barriers, which interlocks them: neither can
// arrive twice on one barrier before the other has passed it.
template <int BV>
struct BoxStore {
    int q4, cg, lane;
    __device__ __forceinline__ bool issuer() const { return BV == 128 || cg == 0; }
    // before the tile is rewritten; `newer_pending`: the issuer has one more recent store group in flight
    // (of the other tile) that may stay in flight
    __device__ __forceinline__ void free_tile(bool newer_pending) const {
        if (issuer() && lane == 0) {
            if (newer_pending)
                tma::wait_read1();
            else
                tma::wait_read();
        }
        __syncwarp();
        if (BV == 64) {
            if (cg == 0)
                bar_arrive(4 + q4, 64);
            else
                bar_sync(4 + q4, 64);
        }
    }
    // after the rows are written and fenced for the async proxy: stores the box (map coordinates x, y, z)
    __device__ __forceinline__ void store(const CUtensorMap *map, int x, int y, int z, uint32_t src) const {
        if (BV == 64) {
            if (cg == 0)
                bar_sync(8 + q4, 64);
            else
                bar_arrive(8 + q4, 64);
        }
        if (issuer() && lane == 0) {
            tma::store3d(map, x, y, z, src);
            tma::commit_group();
        }
    }
};

// Warp-uniform waits for the roles whose work one lane issues (TMA producer, MMA issuer): the whole warp
// runs the role's loop and polls, and lane 0 alone issues, so no lane of the warp sits at a barrier or a
// shuffle while lane 0 works (a lane working alone in a diverged warp was seen to make slow progress).
__device__ __forceinline__ bool uwait(uint32_t bar, uint32_t parity, volatile int *flag, unsigned *err) {
    return __all_sync(0xffffffffu, wait_phase(bar, parity, flag, err));
}
__device__ __forceinline__ bool utest(uint32_t bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_test(bar, parity));
}
__device__ __forceinline__ bool uflag(volatile int *flag) { return __any_sync(0xffffffffu, *flag != 0); }

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

// The intra-GPU split: block z of a launch over N x nseg is segment z % nseg of sequence z / nseg, the
// sequence's whole chunks [cb, cb + sl) with sl = ceil(chunks / nseg) (the affine passes' segments); the
// sequence's first token, length and first chunk row move to the segment's (an empty segment has length 0).
__device__ __forceinline__ void seg_range(int nseg, int seg, long long &tok0, int &len, int &row0) {
    if (nseg <= 1) return;
    const int nc_all = (len + C - 1) / C, sl = (nc_all + nseg - 1) / nseg;
    const int cb = min(nc_all, seg * sl), ce = min(nc_all, cb + sl);
    tok0 += (long long)cb * C;
    row0 += cb;
    len = ce > cb ? min(len - cb * C, (ce - cb) * C) : 0;
}

template <typename T, int BV, bool WRITE_O>
__device__ __forceinline__ void ws_fwd_body(const Geo &geo, const WsP &p, const int vh, const int j, const int nz) {
    using L = Lay<BV, WRITE_O>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const int kind = p.affine ? vh : 0;  // (the affine pass: block x is the kind, the slice is the whole width)
    const int v0 = p.affine ? 0 : vh * BV;
    const int Hv = geo.Hv, Hq = geo.Hq, hq = j / (Hv / Hq);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr bool bf16 = IsBf16<T>::value;
    const int nseg = p.nseg > 1 ? p.nseg : 1, rank = nz / nseg, seg = nz - rank * nseg;
    const int n = geo.sorder ? geo.sorder[rank] : rank;  // (packed batches: the longest sequences start first)
    long long tok0;
    int len, row0;
    geo.seq(n, tok0, len, row0);
    seg_range(nseg, seg, tok0, len, row0);
    const int nc = (len + C - 1) / C;
    volatile int *flag = reinterpret_cast<volatile int *>(smem + L::FLAG);
    float *F = reinterpret_cast<float *>(smem + L::F);
    auto fa = [&](int lc, int which) -> float * { return F + ((lc & 3) * NF + which) * 64; };

    if (tid == 0) {
        umma::mbar_init(sb + L::B_FULL, 1);
        umma::mbar_init(sb + L::B_FULL + 8, 1);
        umma::mbar_init(sb + L::B_EMPTY, 1);
        umma::mbar_init(sb + L::B_EMPTY + 8, 1);
        umma::mbar_init(sb + L::B_FULLL, 1);
        umma::mbar_init(sb + L::B_FULLL + 8, 1);
        // (k and P: released by the MMA warp after the output product and by warp 4 after X)
        umma::mbar_init(sb + L::B_EMPTYL, 2);
        umma::mbar_init(sb + L::B_EMPTYL + 8, 2);
        umma::mbar_init(sb + L::B_PREP, 4);
        umma::mbar_init(sb + L::B_MPW, 1);
        umma::mbar_init(sb + L::B_MPU, 1);
        umma::mbar_init(sb + L::B_MA, 2);
        umma::mbar_init(sb + L::B_EPIA, 4);
        umma::mbar_init(sb + L::B_MB, 1);
        umma::mbar_init(sb + L::B_EPIB, 10);  // the 8 state warps and the 2 -W warps: round A's operands
        umma::mbar_init(sb + L::B_MO, 1);
        umma::mbar_init(sb + L::B_MO + 8, 1);
        umma::mbar_init(sb + L::B_OFREE, 2);
        umma::mbar_init(sb + L::B_OFREE + 8, 2);
        umma::mbar_init(sb + L::B_DONE, 1);
        umma::fence_mbar_init();
        *flag = 0;
    }
    // the zero block between A diag(beta e^G rk) and A diag(beta)
    for (int i = tid; i < 8192 / 16; i += WS_NT) st_v4(sb + L::Z + i * 16, 0u, 0u, 0u, 0u);
    umma::fence_async_smem();
    if (warp == 0) umma::alloc(sb + L::SLOT, 512);
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::SLOT);

    if (warp == 1) {
        // ------------------------------------------------------------ TMA producer
        {
            const bool l0 = lane == 0;
            int issued[2] = {0, 0}, issued_l[2] = {0, 0};
            for (int lc = 0; lc < nc && !uflag(flag); ++lc) {
                const int s = lc & 1;
                const uint32_t st = sb + s * L::ST_BYTES;
                const int t = (int)(tok0 + (long long)lc * C);
                // early group: free once round A of chunk lc - 2 has run
                if (lc >= 2 && !uwait(sb + L::B_EMPTY + 8 * s, ((lc >> 1) - 1) & 1, flag, geo.err)) break;
                const uint32_t fe = sb + L::B_FULL + 8 * s, fl = sb + L::B_FULLL + 8 * s;
                if (l0) tma::expect_tx(fe, (WRITE_O ? 16384u : 0u) + (uint32_t)BV * 128u + 8192u);
                if (WRITE_O) {
                    if (l0) tma::load3d(st + L::ST_Q0, &p.tq, 0, hq, t, fe);
                    if (l0) tma::load3d(st + L::ST_Q1, &p.tq, 64, hq, t, fe);
                }
                if (l0) tma::load3d(st + L::ST_V, &p.tv, v0, j, t, fe);
                if (BV == 128 && l0) tma::load3d(st + L::ST_V + 8192, &p.tv, v0 + 64, j, t, fe);
                if (l0) tma::load3d(st + L::ST_A, &p.ta, 0, j, t, fe);
                ++issued[s];
                // late group: free once round B of chunk lc - 2 has run
                if (lc >= 2 && !uwait(sb + L::B_EMPTYL + 8 * s, ((lc >> 1) - 1) & 1, flag, geo.err)) break;
                if (l0) tma::expect_tx(fl, 16384u + (WRITE_O ? 8192u : 0u));
                if (l0) tma::load3d(st + L::ST_K0, &p.tk, 0, hq, t, fl);
                if (l0) tma::load3d(st + L::ST_K1, &p.tk, 64, hq, t, fl);
                if (WRITE_O && l0) tma::load3d(st + L::ST_P, &p.tp, 0, j, t, fl);
                ++issued_l[s];
                // the next chunk's boxes into L2 now: its loads wait for this stage's turn, a chunk from now
                if (lc + 1 < nc) {
                    const int tn = t + C;
                    if (WRITE_O) {
                        if (l0) tma::prefetch3d(&p.tq, 0, hq, tn);
                        if (l0) tma::prefetch3d(&p.tq, 64, hq, tn);
                        if (l0) tma::prefetch3d(&p.tp, 0, j, tn);
                    }
                    if (l0) tma::prefetch3d(&p.tv, v0, j, tn);
                    if (BV == 128 && l0) tma::prefetch3d(&p.tv, v0 + 64, j, tn);
                    if (l0) tma::prefetch3d(&p.ta, 0, j, tn);
                    if (l0) tma::prefetch3d(&p.tk, 0, hq, tn);
                    if (l0) tma::prefetch3d(&p.tk, 64, hq, tn);
                }
            }
            // let every load in flight land before the block can exit (bounded)
            for (int s = 0; s < 2; ++s) {
                if (issued[s] > 0) umma::mbar_wait(sb + L::B_FULL + 8 * s, (issued[s] - 1) & 1, 4000000L);
                if (issued_l[s] > 0) umma::mbar_wait(sb + L::B_FULLL + 8 * s, (issued_l[s] - 1) & 1, 4000000L);
            }
        }
    } else if (warp == 0) {
        // ------------------------------------------------------------ MMA issue
        {
            const bool l0 = lane == 0;
            const uint32_t id_w = umma::idesc(128, 128, bf16, false, true);
            const uint32_t id_bv = umma::idesc(128, BV, bf16, false, true);   // K-major A, MN-major B
            const uint32_t id_mn = umma::idesc(128, BV, bf16, true, true);    // MN-major A and B
            const uint64_t dZAKG = umma::desc(sb + L::Z, 16, 1024), dABZ = umma::desc(sb + L::AB, 16, 1024);
            const uint64_t dH = umma::desc(sb + L::H, 16384, 1024);
            const uint64_t dDL = umma::desc(sb + L::DL, 8192, 1024);
            auto issue_w = [&](int lc) {  // W of chunk lc
                const uint32_t st = sb + (lc & 1) * L::ST_BYTES;
                const uint64_t bk = umma::desc(st + L::ST_K0, L::LBO_K, 1024);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) if (l0) umma::mma(tmem + L::T_W, dZAKG + ks * 2, bk + ks * 128, id_w, ks > 0);
            };
            auto issue_u = [&](int lc) {  // U of chunk lc (also zeroes the output lanes 64..127)
                const uint32_t st = sb + (lc & 1) * L::ST_BYTES;
                const uint64_t bv = umma::desc(st + L::ST_V, 8192, 1024);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    if (l0) umma::mma(tmem + ((lc & 1) ? L::T_D1 : L::T_D0), dABZ + ks * 2, bv + ks * 128, id_bv, ks > 0);
            };
            bool ok = true;
            if (nc > 0) {
                ok = uwait(sb + L::B_PREP, 0, flag, geo.err) && uwait(sb + L::B_FULL, 0, flag, geo.err) &&
                     uwait(sb + L::B_FULLL, 0, flag, geo.err);
                umma::fence_after();
                if (ok) {
                    issue_w(0);
                    if (l0) umma::commit(sb + L::B_MPW);
                    issue_u(0);
                    if (l0) umma::commit(sb + L::B_MPU);
                }
            }
            for (int lc = 0; lc < nc && ok; ++lc) {
                const int b = lc & 1;
                const uint32_t st = sb + b * L::ST_BYTES;
                const uint32_t tD = b ? L::T_D1 : L::T_D0;
                // round A: needs -W (rows above Q) and the state tile, both announced on B_EPIB (one barrier to pass)
                if (!(ok = uwait(sb + L::B_EPIB, lc & 1, flag, geo.err)))
                    break;
                umma::fence_after();
                {
                    const uint64_t aqw = umma::desc(st + L::ST_W0, 16, 1024);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        if (l0) umma::mma(tmem + tD, aqw + ((((ks >> 2) * 16384) + (ks & 3) * 32) >> 4), dH + ks * 128, id_bv,
                                  true);
                }
                if (l0) umma::commit(sb + L::B_MA);
                if (l0) mbar_arrive(sb + L::B_MA);
                if (l0) umma::commit(sb + L::B_EMPTY + 8 * b);  // q, v and A of this chunk are done
                // round B as soon as Delta is in shared memory; the next chunk's W group goes in whenever
                // its inputs are ready, its U group (needed only by the next round A) after round B
                const bool next = lc + 1 < nc;
                bool b_done = false, w_done = !next, u_done = !next;
                for (long it = 0; !(b_done && w_done && u_done); ++it) {
                    if (!b_done && utest(sb + L::B_EPIA, lc & 1)) {
                        // round B's output product (its X product is issued by the Delta-row warps themselves)
                        umma::fence_after();
                        const uint64_t ap = umma::desc(st + L::ST_A, 16, 1024);
                        if (WRITE_O) {
                            // P Delta into its own columns: the output epilogue scales the Q h rows alone
                            const uint32_t tPD = b ? L::T_PD1 : L::T_PD0;
#pragma unroll
                            for (int ks = 0; ks < 4; ++ks) if (l0) umma::mma(tmem + tPD, ap + ks * 2, dDL + ks * 128, id_bv, ks > 0);
                        }
                        if (l0) umma::commit(sb + L::B_EMPTYL + 8 * b);  // k and P are done
                        if (l0) umma::commit(sb + L::B_MO + 8 * b);
                        b_done = true;
                        continue;
                    }
                    if (!w_done && utest(sb + L::B_PREP, (lc + 1) & 1) &&
                        utest(sb + L::B_FULLL + 8 * (b ^ 1), ((lc + 1) >> 1) & 1)) {
                        umma::fence_after();
                        issue_w(lc + 1);
                        if (l0) umma::commit(sb + L::B_MPW);
                        w_done = true;
                        continue;
                    }
                    if (!u_done && w_done && b_done &&
                        (!WRITE_O || lc < 1 || utest(sb + L::B_OFREE + 8 * (b ^ 1), ((lc - 1) >> 1) & 1))) {
                        umma::fence_after();
                        issue_u(lc + 1);
                        if (l0) umma::commit(sb + L::B_MPU);
                        u_done = true;
                        continue;
                    }
                    if ((it & 127) == 127 && uflag(flag)) {
                        ok = false;
                        break;
                    }
                    if (it > kWaitPolls) {
                        raise_error(geo.err, GDR_ERR_TIMEOUT);
                        *flag = 1;
                        ok = false;
                        break;
                    }
                }
            }
            // every MMA issued so far completes before TMEM is released
            if (l0) umma::commit(sb + L::B_DONE);
            umma::mbar_wait(sb + L::B_DONE, 0, 4000000L);
        }
    } else if (warp >= 12) {
        // ------------------------------------------------------------ preparation (128 threads)
        const int at = (warp - 12) * 32 + lane;  // 0..127
        float x0 = 0.f, x1 = 0.f;  // prefetched: G, rq (threads 0..63) or beta, rk (64..127)
        auto fetch = [&](int lc) {
            const int valid = min(C, len - lc * C);
            const int r = at & 63;
            x0 = 0.f;
            x1 = 1.f;
            if (r < valid) {
                const long long ti = (tok0 + (long long)lc * C + r) * Hv + j;
                if (at < 64) {
                    x0 = p.g_cs[ti];
                    if (p.l2norm && WRITE_O) x1 = p.rq[ti];
                } else {
                    x0 = load_gate<T>(p.beta, ti, p.gate_f32);
                    if (p.l2norm) x1 = p.rk[ti];
                }
            }
        };
        if (nc > 0) fetch(0);
        for (int lc = 0; lc < nc; ++lc) {
            const int s = lc & 1;
            const uint32_t st = sb + s * L::ST_BYTES;
            const int valid = min(C, len - lc * C);
            if (at < 64) {
                fa(lc, FG)[at] = x0;
                fa(lc, FRQ)[at] = x1;
            } else {
                fa(lc, FB)[at - 64] = x0;
                fa(lc, FRK)[at - 64] = x1;
            }
            if (lc + 1 < nc) fetch(lc + 1);
            asm volatile("bar.sync 1, 128;\n" ::: "memory");
            if (at < 64) {
                const int r = at;
                const bool ok = r < valid;
                const float gr = fa(lc, FG)[r], Gl = fa(lc, FG)[valid - 1];
                const float rq = fa(lc, FRQ)[r], rk = fa(lc, FRK)[r], be = fa(lc, FB)[r];
                const float eg = __expf(gr);
                fa(lc, FCQ)[r] = ok ? p.scale * rq * eg : 0.f;
                fa(lc, FCK)[r] = ok ? rk * __expf(Gl - gr) : 0.f;
                fa(lc, FAKG)[r] = ok ? be * eg * rk : 0.f;
                fa(lc, FAB)[r] = (ok && kind == 0) ? be : 0.f;  // (identity-start affine kind: U = 0)
            }
            // the stage's tiles, and the previous chunk's W and U groups done with the scaled copies of A
            // (warp 14 polls the barriers and the four prep warps share the result through a hardware barrier:
            // fewer warps polling mbarriers on one scheduler see their phases sooner)
            bool ok = true;
            if (warp == 14) {
                ok = warp_wait(sb + L::B_FULL + 8 * s, (lc >> 1) & 1, flag, geo.err, lane);
                if (ok && lc > 0) ok = warp_wait(sb + L::B_MPU, (lc - 1) & 1, flag, geo.err, lane);
            }
            if (!group_and(ok, 1, 128)) break;
            {
                // A diag(beta e^G rk) and A diag(beta): thread -> row at/2, 32 columns; rows past the end are
                // zero.  Every shared load is issued before the first store (the stores are ordered asm).
                const int r = at >> 1, c0 = (at & 1) * 32;
                const bool okr = r < valid;
                const float4 *fk4 = reinterpret_cast<const float4 *>(fa(lc, FAKG) + c0);
                const float4 *fb4 = reinterpret_cast<const float4 *>(fa(lc, FAB) + c0);
                uint4 u[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) u[c] = umma::ld_shared_v4(st + L::ST_A + umma::off(r, c0 + c * 8, 0));
                float fkv[32], fbv[32];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 a = fk4[i], bq = fb4[i];
                    fkv[4 * i] = a.x, fkv[4 * i + 1] = a.y, fkv[4 * i + 2] = a.z, fkv[4 * i + 3] = a.w;
                    fbv[4 * i] = bq.x, fbv[4 * i + 1] = bq.y, fbv[4 * i + 2] = bq.z, fbv[4 * i + 3] = bq.w;
                }
                uint32_t wk[16], wb[16];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t w[4] = {u[c].x, u[c].y, u[c].z, u[c].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 x = Elt<T>::unpack(w[e]);
                        const int i = c * 8 + 2 * e;
                        wk[c * 4 + e] = Elt<T>::pack(okr ? x.x * fkv[i] : 0.f, okr ? x.y * fkv[i + 1] : 0.f);
                        wb[c * 4 + e] = Elt<T>::pack(okr ? x.x * fbv[i] : 0.f, okr ? x.y * fbv[i + 1] : 0.f);
                    }
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t o = umma::off(r, c0 + c * 8, 0);
                    st_v4(sb + L::AKG + o, wk[4 * c], wk[4 * c + 1], wk[4 * c + 2], wk[4 * c + 3]);
                    st_v4(sb + L::AB + o, wb[4 * c], wb[4 * c + 1], wb[4 * c + 2], wb[4 * c + 3]);
                }
            }
            umma::fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(sb + L::B_PREP);
        }
    } else if (warp >= 4 && warp < 12) {
        // ------------------------------------------------------------ state (256 threads)
        const int sw = warp - 4, q4 = warp & 3, cg = sw >> 2;
        const int d = q4 * 32 + lane;  // TMEM lane: key row of h; for q4 < 2 also token row d of Delta
        constexpr int HW = BV / 2;     // value columns per thread
        const int cb0 = cg * HW;
        const long long st_base = ((long long)n * Hv + j) * DK * DV;
        const long long seg_base = (((long long)n * Hv + j) * nseg + seg) * DK * DV;
        float hS[HW];
#pragma unroll
        for (int i = 0; i < HW; ++i) {
            const int e = v0 + cb0 + i;
            if (p.affine)
                hS[i] = (kind == 1 && e == d) ? 1.f : 0.f;
            else if (p.seg_start)
                hS[i] = p.seg_start[seg_base + (long long)e * DK + d];
            else if (p.h0)
                hS[i] = p.h0[st_base + (p.v_first ? (long long)e * DK + d : (long long)d * DV + e)];
            else
                hS[i] = 0.f;
        }
        const BoxStore<BV> box{q4, cg, lane};
        const int bx = cb0 & ~63;  // first column of the stored box that holds this warp's columns
        // the state before chunk lcn into the operand tile (and, with tma_h, on to h as a TMA box)
        auto write_h = [&](int lcn) {
            // (a Delta-row warp's newer group in flight is this chunk's Delta box)
            if (p.tma_h) box.free_tile(q4 < 2 && p.tma_delta && lcn > 0);
#pragma unroll
            for (int i = 0; i < HW; i += 16) {
                const int col = cb0 + i;
                store_row16<T>(sb + L::H + (col >> 6) * 16384, d, col & 63, hS + i);
            }
            umma::fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(sb + L::B_EPIB);
            if (p.tma_h && lcn < nc)
                box.store(&p.th, v0 + bx, q4 * 32, (row0 + lcn) * Hv + j, sb + L::H + (bx >> 6) * 16384 + q4 * 4096);
        };
        write_h(0);
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
            if (p.h && !p.tma_h) {
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
            bool okw = true;  // every state warp reaches the hardware barriers below, failed or not
            // round A's barrier: polled by warp 5 alone and shared with the other Delta-row warps (4, 8, 9)
            // through a hardware barrier, so that the MMA thread is the only warp polling on its scheduler
            if (q4 < 2) {
                if (warp == 5) okw = warp_wait(sb + L::B_MA, lc & 1, flag, geo.err, lane);
                okw = group_and(okw, 3, 128);
            }
            if (q4 < 2 && okw) {
                // Delta rows (lanes 0..63): Delta for the output product, diag(rk e^{Gl-G}) Delta for X
                umma::fence_after();
                const int sr = d;
                const float ck = fa(lc, FCK)[sr];
                // the Delta box stored last chunk has been read (the state box stored since may stay in flight)
                if (p.tma_delta) box.free_tile(p.tma_h);
                constexpr int NB = HW < 32 ? HW : 32;  // columns per TMEM load batch
#pragma unroll
                for (int i0 = 0; i0 < HW; i0 += NB) {
                float xa[NB];
#pragma unroll
                for (int i = 0; i < NB; i += 16) umma::ld16(umma::taddr(tmem, q4 * 32, tD + cb0 + i0 + i), xa + i);
                umma::ld_wait();
#pragma unroll
                for (int i = 0; i < NB; i += 16) {
                    float *x = xa + i, y[16];
                    const int col = cb0 + i0 + i;
#pragma unroll
                    for (int u = 0; u < 16; ++u) y[u] = x[u] * ck;
                    if (WRITE_O || p.tma_delta) store_row16<T>(sb + L::DL + (col >> 6) * 8192, sr, col & 63, x);
                    store_row16<T>(sb + L::DT + (col >> 6) * 8192, sr, col & 63, y);
                    if (p.delta && !p.tma_delta) {
                        T *dr = static_cast<T *>(p.delta) + (((long long)(row0 + lc) * Hv + j) * C + sr) * DV + v0 + col;
                        *reinterpret_cast<uint4 *>(dr) =
                            make_uint4(Elt<T>::pack(x[0], x[1]), Elt<T>::pack(x[2], x[3]), Elt<T>::pack(x[4], x[5]),
                                       Elt<T>::pack(x[6], x[7]));
                        *reinterpret_cast<uint4 *>(dr + 8) =
                            make_uint4(Elt<T>::pack(x[8], x[9]), Elt<T>::pack(x[10], x[11]),
                                       Elt<T>::pack(x[12], x[13]), Elt<T>::pack(x[14], x[15]));
                    }
                }
                }
                umma::fence_before();
                umma::fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(sb + L::B_EPIA);
                // round B's X = K^T (diag(ck) Delta) goes in from here, not from the MMA warp: the four Delta-row
                // warps meet at a hardware barrier and warp 4 issues it, which spares the state's critical path
                // the MMA warp's late view of B_EPIA
                asm volatile("bar.sync 3, 128;\n" ::: "memory");
                if (warp == 4) {
                    if (lane == 0) {
                        umma::fence_after();
                        const uint32_t stx = sb + (lc & 1) * L::ST_BYTES;
                        const uint64_t akt = umma::desc(stx + L::ST_K0, L::LBO_K, 1024);
                        const uint64_t dDTx = umma::desc(sb + L::DT, 8192, 1024);
                        const uint32_t idx = umma::idesc(128, BV, IsBf16<T>::value, true, true);
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) umma::mma(tmem + L::T_X, akt + ks * 128, dDTx + ks * 128, idx, ks > 0);
                        umma::commit(sb + L::B_MB);
                        umma::commit(sb + L::B_EMPTYL + 8 * (lc & 1));
                    }
                    __syncwarp();
                }
                if (p.tma_delta)
                    box.store(&p.tdl, v0 + bx, q4 * 32, (row0 + lc) * Hv + j, sb + L::DL + (bx >> 6) * 8192 + q4 * 4096);
            }
            // round B's barrier is polled by one warp (5, after its Delta rows) and passed on to the other state
            // warps by a hardware barrier: warps that polled it themselves from the schedulers shared with
            // other polling warps were seen to pass it several hundred cycles late
            if (warp == 5 && okw) okw = warp_wait(sb + L::B_MB, lc & 1, flag, geo.err, lane);
            if (!group_and(okw, 2, 256)) break;  // the eight state warps: all go on, or all leave
            umma::fence_after();
            {
                constexpr int NB = HW < 32 ? HW : 32;
#pragma unroll
                for (int i0 = 0; i0 < HW; i0 += NB) {
                    float xb[NB];
#pragma unroll
                    for (int i = 0; i < NB; i += 16) umma::ld16(umma::taddr(tmem, q4 * 32, L::T_X + cb0 + i0 + i), xb + i);
                    umma::ld_wait();
#pragma unroll
                    for (int i = 0; i < NB; ++i) hS[i0 + i] = fmaf(egl, hS[i0 + i], xb[i]);
                }
            }
            umma::fence_before();
            write_h(lc + 1);
        }
        if (lane == 0 && (p.tma_h || p.tma_delta)) tma::wait_all();  // the stored boxes are complete (issuers)
        if (!*flag && p.affine) {
#pragma unroll
            for (int i = 0; i < HW; ++i) p.seg_end[kind][seg_base + (long long)(v0 + cb0 + i) * DK + d] = hS[i];
        } else if (!*flag && p.fin && seg == nseg - 1) {
#pragma unroll
            for (int i = 0; i < HW; ++i) {
                const int e = v0 + cb0 + i;
                p.fin[st_base + (p.v_first ? (long long)e * DK + d : (long long)d * DV + e)] = hS[i];
            }
        }
    } else {
        // ------------------------------------------------------------ -W and output rows (warps 2, 3)
        const int r = (warp - 2) * 32 + lane;  // token row; TMEM lane 64 + r
        const int lb = 32 * (warp & 3);
        auto out_rows = [&](int lc) -> bool {
            const int b = lc & 1;
            const int valid = min(C, len - lc * C);
            if (!warp_wait(sb + L::B_MO + 8 * b, (lc >> 1) & 1, flag, geo.err, lane)) return false;
            umma::fence_after();
            const uint32_t tD = b ? L::T_D1 : L::T_D0, tPD = b ? L::T_PD1 : L::T_PD0;
            const float cq = fa(lc, FCQ)[r];  // scale rq e^G of this row (0 past the end)
            T *orow = static_cast<T *>(p.o) + ((tok0 + (long long)lc * C + r) * Hv + j) * geo.V + v0;
            // a full chunk's rows leave through the staging tile, this warp's 32 rows as one TMA box (scattered
            // row stores would crowd the memory instruction queue of the schedulers the state warps share);
            // a ragged chunk's rows are stored directly (its tail rows belong to the next sequence)
            const bool staged = valid == C;
            const uint32_t ost = sb + L::OST;
            if (staged) {
                if (lane == 0) tma::wait_read();  // the previous box has left the staging tile
                __syncwarp();
            }
#pragma unroll
            for (int c = 0; c < BV; c += 16) {
                float x[16], y[16];
                umma::ld16(umma::taddr(tmem, lb, tD + c), x);
                umma::ld16(umma::taddr(tmem, lb, tPD + c), y);
                umma::ld_wait();  // (one 16-column slice at a time keeps the warp's registers low)
#pragma unroll
                for (int u = 0; u < 16; ++u) x[u] = fmaf(cq, x[u], y[u]);  // o = diag(scale rq e^G) Q h + P Delta
                const uint32_t w0 = Elt<T>::pack(x[0], x[1]), w1 = Elt<T>::pack(x[2], x[3]),
                               w2 = Elt<T>::pack(x[4], x[5]), w3 = Elt<T>::pack(x[6], x[7]),
                               w4 = Elt<T>::pack(x[8], x[9]), w5 = Elt<T>::pack(x[10], x[11]),
                               w6 = Elt<T>::pack(x[12], x[13]), w7 = Elt<T>::pack(x[14], x[15]);
                if (staged) {
                    st_v4(ost + (uint32_t)(c >> 6) * 8192u + umma::off(r, (c & 63), 0), w0, w1, w2, w3);
                    st_v4(ost + (uint32_t)(c >> 6) * 8192u + umma::off(r, (c & 63) + 8, 0), w4, w5, w6, w7);
                } else if (r < valid) {
                    if (v0 + c < geo.V) *reinterpret_cast<uint4 *>(orow + c) = make_uint4(w0, w1, w2, w3);
                    if (v0 + c + 8 < geo.V) *reinterpret_cast<uint4 *>(orow + c + 8) = make_uint4(w4, w5, w6, w7);
                }
            }
            umma::fence_before();
            if (staged) umma::fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(sb + L::B_OFREE + 8 * b);
                if (staged) {
                    const int t0 = (int)(tok0 + (long long)lc * C) + (warp - 2) * 32;
#pragma unroll
                    for (int cb = 0; cb < BV; cb += 64)
                        if (v0 + cb < geo.V)
                            tma::store3d(&p.to, v0 + cb, j, t0, ost + (uint32_t)(cb >> 6) * 8192u + (warp - 2) * 4096);
                    tma::commit_group();
                }
            }
            return true;
        };
        bool ok = true;
        for (int lc = 0; lc < nc && ok; ++lc) {
            if (!warp_wait(sb + L::B_MPW, lc & 1, flag, geo.err, lane)) break;
            umma::fence_after();
            {
                // -W row r (128 key columns) into the rows above Q of this chunk's stage
                const uint32_t st = sb + (lc & 1) * L::ST_BYTES;
#pragma unroll
                for (int c = 0; c < 128; c += 64) {
                    float x[64];
#pragma unroll
                    for (int u = 0; u < 64; u += 16) umma::ld16(umma::taddr(tmem, lb, L::T_W + c + u), x + u);
                    umma::ld_wait();
#pragma unroll
                    for (int u = 0; u < 64; ++u) x[u] = -x[u];
                    const uint32_t blk = st + (c < 64 ? L::ST_W0 : L::ST_W1);
#pragma unroll
                    for (int u = 0; u < 64; u += 16) store_row16<T>(blk, r, u, x + u);
                }
            }
            umma::fence_before();
            umma::fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(sb + L::B_EPIB);  // (-W of this chunk: the other half of round A's inputs)
            if (WRITE_O && lc > 0) ok = out_rows(lc - 1);
        }
        if (WRITE_O && ok && nc > 0) out_rows(nc - 1);
        if (WRITE_O && lane == 0) tma::wait_all();  // the output boxes are complete
    }

    umma::fence_before();
    __syncthreads();
    if (warp == 0) umma::dealloc(tmem, 512);
}

template <typename T, int BV, bool WRITE_O>
__global__ void __launch_bounds__(WS_NT, 1) chain_ws_kernel(Geo geo, const __grid_constant__ WsP p) {
    griddep_launch_next();
    griddep_wait();
    ws_fwd_body<T, BV, WRITE_O>(geo, p, blockIdx.x, blockIdx.y, blockIdx.z);
}

// ============================================================================ reverse chain
//
// The gradient of the state, dh [K x V], runs the chunks backwards; its value columns are independent,
// so one CTA of 512 threads owns one (sequence, value head, BV-wide slice of the value columns): BV = 64
// (two CTAs per head) when the forward's states are at hand and the chain runs alone, BV = 128 beside the
// forward recompute.  The warp roles are the forward's.  With dh' the gradient after chunk c,
// P = scale (q^ k^T o Gamma) (lower), Q~ = diag(scale rq e^G) Q and W = A diag(beta e^G rk) K:
//
//   dDelta = diag(rk e^{Gl-G}) (K dh') + P^T dO                     [64 x V]
//   dh     = e^{Gl} dh' + Q~^T dO - W^T dDelta                        [K x V]
//
//   state-independent:  P^T dO -> T_P, Q~^T dO -> T_Y (the base of round B), W -> T_W (the -W epilogue)
//   round A:  E = [K ; .] dh'                  (lanes 0..63)           M=128, N=BV, K=128
//   round B:  T_Y += (-W)^T dDelta                                     M=128, N=BV, K=64
// It stores dh' of every chunk (the gradient after the chunk) and dDelta for the per-chunk gradients;
// the last dh is dh0.

struct RLay {
    // stage: [Q~ b0 | Q~ b1 | K b0 | K b1 | dO b0 | dO b1 | A | P], 8 KB blocks of 64 rows x 128 B
    static constexpr uint32_t ST_Q0 = 0, ST_K0 = 16384, ST_DO = 32768, ST_A = 49152, ST_P = 57344,
                              ST_BYTES = 65536;
    static constexpr uint32_t WS = 2 * ST_BYTES;  // -W [64 s][128 d]: two 8 KB blocks (one buffer)
    static constexpr uint32_t Z = WS + 16384;     // zeros, then A diag(beta e^G rk): [0 ; A diag(..)]
    static constexpr uint32_t AKG = Z + 8192;
    static constexpr uint32_t DL = AKG + 8192;    // dDelta [64 s][128]: two 8 KB blocks
    static constexpr uint32_t H = DL + 16384;     // dh' [128 d][128]: two 16 KB blocks
    static constexpr uint32_t F = H + 32768;
    static constexpr uint32_t BAR = F + 4 * NF * 256;
    static constexpr uint32_t B_FULL = BAR, B_EMPTY = BAR + 16, B_PREP = BAR + 32,
                              B_MPW = BAR + 48, B_MA = BAR + 56, B_EPIA = BAR + 64, B_MB = BAR + 72,
                              B_EPIB = BAR + 80, B_DONE = BAR + 88;
    // the preparation is released in two steps: B_PREP (A diag(beta e^G rk) and P's rows past the end: P^T dO
    // and W may go) and B_PREPQ + 8 (c & 1) (Q~ of chunk step c in place: Q~^T dO may go).  B_PREPQ is a ring of
    // two so that the preparation, which runs ahead, can never complete a phase its waiter has not yet seen.
    static constexpr uint32_t B_PREPQ = BAR + 96;
    static constexpr uint32_t SLOT = BAR + 112, FLAG = SLOT + 4, USED = FLAG + 12;
    static constexpr uint32_t BYTES = USED + 1024;
    static constexpr uint32_t T_W = 0, T_E = 128, T_P = 256, T_Y = 384;
};
static_assert(RLay::BYTES <= 232448, "shared memory");

struct RevP {
    CUtensorMap tq, tk, tdo, tp, ta;  // [tokens][heads][cols] maps, boxes 64 x 1 x 64
    const float *g_cs, *rq, *rk, *dht;
    const float *seg_start;  // optional end-of-segment gradients, transposed [N,Hv,nseg,V,K] fp32 (replaces dht)
    int nseg;                // segments per sequence (1 = none): grid z = N x nseg
    float *seg_end;          // optional: every segment's gradient at its start, transposed [N,Hv,nseg,V,K] fp32
                             // (the split's zero-start reverse pass; dh0 is then not written)
    const void *beta;
    void *dhn;     // [rows,Hv,K,V]: the gradient after every chunk
    void *ddelta;  // [rows,Hv,64,V]
    float *dh0;
    bool gate_f32, l2norm, v_first;
    float scale;
    // dH' and dDelta leave by TMA store from the bf16 tiles in shared memory (each state warp its own
    // 32-row x 64-column box); boxes 64 x 32 x 1
    CUtensorMap tdh, tdd;
};

template <typename T, int BV>
__device__ __forceinline__ void ws_rev_body(const Geo &geo, const RevP &p, const int vh, const int j, const int nz) {
    using L = RLay;
    const int v0 = vh * BV;  // this block's value columns v0 .. v0+BV-1
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const int Hv = geo.Hv, Hq = geo.Hq, hq = j / (Hv / Hq);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr bool bf16 = IsBf16<T>::value;
    const int nseg = p.nseg > 1 ? p.nseg : 1, rank = nz / nseg, seg = nz - rank * nseg;
    const int n = geo.sorder ? geo.sorder[rank] : rank;  // (packed batches: the longest sequences start first)
    long long tok0;
    int len, row0;
    geo.seq(n, tok0, len, row0);
    seg_range(nseg, seg, tok0, len, row0);
    const int nc = (len + C - 1) / C;
    auto chunk_of = [&](int lc) { return nc - 1 - lc; };
    volatile int *flag = reinterpret_cast<volatile int *>(smem + L::FLAG);
    float *F = reinterpret_cast<float *>(smem + L::F);
    auto fa = [&](int lc, int which) -> float * { return F + ((lc & 3) * NF + which) * 64; };

    if (tid == 0) {
        umma::mbar_init(sb + L::B_FULL, 1);
        umma::mbar_init(sb + L::B_FULL + 8, 1);
        umma::mbar_init(sb + L::B_EMPTY, 1);
        umma::mbar_init(sb + L::B_EMPTY + 8, 1);
        umma::mbar_init(sb + L::B_PREP, 4);
        umma::mbar_init(sb + L::B_PREPQ, 4);
        umma::mbar_init(sb + L::B_PREPQ + 8, 4);
        umma::mbar_init(sb + L::B_MPW, 1);
        umma::mbar_init(sb + L::B_MA, 2);  // the commit, and the issuing thread's own arrival
        umma::mbar_init(sb + L::B_EPIA, 6);  // the 4 dDelta-row warps and the 2 -W warps: round B's operands
        umma::mbar_init(sb + L::B_MB, 1);
        umma::mbar_init(sb + L::B_EPIB, 8);
        umma::mbar_init(sb + L::B_DONE, 1);
        umma::fence_mbar_init();
        *flag = 0;
    }
    for (int i = tid; i < 8192 / 16; i += WS_NT) st_v4(sb + L::Z + i * 16, 0u, 0u, 0u, 0u);
    umma::fence_async_smem();
    if (warp == 0) umma::alloc(sb + L::SLOT, 512);
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::SLOT);

    if (warp == 1) {
        // ------------------------------------------------------------ TMA producer
        {
            const bool l0 = lane == 0;
            int issued[2] = {0, 0};
            for (int lc = 0; lc < nc && !uflag(flag); ++lc) {
                const int s = lc & 1;
                if (lc >= 2 && !uwait(sb + L::B_EMPTY + 8 * s, ((lc >> 1) - 1) & 1, flag, geo.err)) break;
                const uint32_t st = sb + s * L::ST_BYTES, full = sb + L::B_FULL + 8 * s;
                const int t = (int)(tok0 + (long long)chunk_of(lc) * C);
                if (l0) tma::expect_tx(full, 49152u + (uint32_t)BV * 128u);
                if (l0) tma::load3d(st + L::ST_Q0, &p.tq, 0, hq, t, full);
                if (l0) tma::load3d(st + L::ST_Q0 + 8192, &p.tq, 64, hq, t, full);
                if (l0) tma::load3d(st + L::ST_K0, &p.tk, 0, hq, t, full);
                if (l0) tma::load3d(st + L::ST_K0 + 8192, &p.tk, 64, hq, t, full);
                if (l0) tma::load3d(st + L::ST_DO, &p.tdo, v0, j, t, full);
                if (BV == 128 && l0) tma::load3d(st + L::ST_DO + 8192, &p.tdo, v0 + 64, j, t, full);
                if (l0) tma::load3d(st + L::ST_A, &p.ta, 0, j, t, full);
                if (l0) tma::load3d(st + L::ST_P, &p.tp, 0, j, t, full);
                ++issued[s];
                // the next chunk's boxes into L2 now: its loads wait for this stage's turn, a chunk from now
                if (lc + 1 < nc) {
                    const int tn = (int)(tok0 + (long long)chunk_of(lc + 1) * C);
                    if (l0) tma::prefetch3d(&p.tq, 0, hq, tn);
                    if (l0) tma::prefetch3d(&p.tq, 64, hq, tn);
                    if (l0) tma::prefetch3d(&p.tk, 0, hq, tn);
                    if (l0) tma::prefetch3d(&p.tk, 64, hq, tn);
                    if (l0) tma::prefetch3d(&p.tdo, v0, j, tn);
                    if (BV == 128 && l0) tma::prefetch3d(&p.tdo, v0 + 64, j, tn);
                    if (l0) tma::prefetch3d(&p.ta, 0, j, tn);
                    if (l0) tma::prefetch3d(&p.tp, 0, j, tn);
                }
            }
            for (int s = 0; s < 2; ++s)
                if (issued[s] > 0) umma::mbar_wait(sb + L::B_FULL + 8 * s, (issued[s] - 1) & 1, 4000000L);
        }
    } else if (warp == 0) {
        // ------------------------------------------------------------ MMA issue
        {
            const bool l0 = lane == 0;
            const uint32_t id_kmn = umma::idesc(128, 128, bf16, false, true);  // K-major A, MN-major B (W)
            const uint32_t id_kbv = umma::idesc(128, BV, bf16, false, true);   // the same, N = BV
            const uint32_t id_mn = umma::idesc(128, BV, bf16, true, true);     // MN-major A and B, N = BV
            const uint64_t dZAKG = umma::desc(sb + L::Z, 16, 1024), dH = umma::desc(sb + L::H, 16384, 1024);
            const uint64_t dWS = umma::desc(sb + L::WS, 8192, 1024), dDL = umma::desc(sb + L::DL, 8192, 1024);
            auto issue_pw = [&](int lc) {  // P^T dO and W of chunk lc
                const uint32_t st = sb + (lc & 1) * L::ST_BYTES;
                const uint64_t ap = umma::desc(st + L::ST_P, 8192, 1024), bdo = umma::desc(st + L::ST_DO, 8192, 1024);
                const uint64_t bk = umma::desc(st + L::ST_K0, 8192, 1024);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) if (l0) umma::mma(tmem + L::T_P, ap + ks * 128, bdo + ks * 128, id_mn, ks > 0);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) if (l0) umma::mma(tmem + L::T_W, dZAKG + ks * 2, bk + ks * 128, id_kmn, ks > 0);
                if (l0) umma::commit(sb + L::B_MPW);
            };
            bool ok = true;
            if (nc > 0) {
                ok = uwait(sb + L::B_PREP, 0, flag, geo.err) && uwait(sb + L::B_FULL, 0, flag, geo.err);
                umma::fence_after();
                if (ok) issue_pw(0);
            }
            for (int lc = 0; lc < nc && ok; ++lc) {
                const int b = lc & 1;
                const uint32_t st = sb + b * L::ST_BYTES;
                // round A on the state tile
                if (!(ok = uwait(sb + L::B_EPIB, lc & 1, flag, geo.err))) break;
                umma::fence_after();
                {
                    const uint64_t ak = umma::desc(st + L::ST_K0, 16, 1024);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        if (l0) umma::mma(tmem + L::T_E, ak + ((((ks >> 2) * 8192) + (ks & 3) * 32) >> 4), dH + ks * 128, id_kbv,
                                  ks > 0);
                }
                if (l0) umma::commit(sb + L::B_MA);
                if (l0) mbar_arrive(sb + L::B_MA);
                // Q~^T dO, the base that round B adds to (Q~ of this chunk step in place)
                if (!(ok = uwait(sb + L::B_PREPQ + 8 * b, (lc >> 1) & 1, flag, geo.err))) break;
                umma::fence_after();
                {
                    const uint64_t aq = umma::desc(st + L::ST_Q0, 8192, 1024), bdo = umma::desc(st + L::ST_DO, 8192, 1024);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) if (l0) umma::mma(tmem + L::T_Y, aq + ks * 128, bdo + ks * 128, id_mn, ks > 0);
                }
                // round B: needs dDelta and -W, both announced on B_EPIA (one barrier to pass)
                if (!(ok = uwait(sb + L::B_EPIA, lc & 1, flag, geo.err)))
                    break;
                umma::fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) if (l0) umma::mma(tmem + L::T_Y, dWS + ks * 128, dDL + ks * 128, id_mn, true);
                if (l0) umma::commit(sb + L::B_MB);
                if (l0) umma::commit(sb + L::B_EMPTY + 8 * b);
                if (lc + 1 < nc) {
                    // (B_PREP implies the stage's tiles: the preparation waited for them before its arrival)
                    if (!(ok = uwait(sb + L::B_PREP, (lc + 1) & 1, flag, geo.err)))
                        break;
                    umma::fence_after();
                    issue_pw(lc + 1);
                }
            }
            if (l0) umma::commit(sb + L::B_DONE);
            umma::mbar_wait(sb + L::B_DONE, 0, 4000000L);
        }
    } else if (warp >= 12) {
        // ------------------------------------------------------------ preparation (128 threads)
        const int at = (warp - 12) * 32 + lane;
        float x0 = 0.f, x1 = 0.f;
        auto fetch = [&](int lc) {
            const int c = chunk_of(lc);
            const int valid = min(C, len - c * C);
            const int r = at & 63;
            x0 = 0.f;
            x1 = 1.f;
            if (r < valid) {
                const long long ti = (tok0 + (long long)c * C + r) * Hv + j;
                if (at < 64) {
                    x0 = p.g_cs[ti];
                    if (p.l2norm) x1 = p.rq[ti];
                } else {
                    x0 = load_gate<T>(p.beta, ti, p.gate_f32);
                    if (p.l2norm) x1 = p.rk[ti];
                }
            }
        };
        if (nc > 0) fetch(0);
        for (int lc = 0; lc < nc; ++lc) {
            const int s = lc & 1;
            const uint32_t st = sb + s * L::ST_BYTES;
            const int valid = min(C, len - chunk_of(lc) * C);
            if (at < 64) {
                fa(lc, FG)[at] = x0;
                fa(lc, FRQ)[at] = x1;
            } else {
                fa(lc, FB)[at - 64] = x0;
                fa(lc, FRK)[at - 64] = x1;
            }
            if (lc + 1 < nc) fetch(lc + 1);
            asm volatile("bar.sync 1, 128;\n" ::: "memory");
            if (at < 64) {
                const int r = at;
                const bool okr = r < valid;
                const float gr = fa(lc, FG)[r], Gl = fa(lc, FG)[valid - 1];
                const float rq = fa(lc, FRQ)[r], rk = fa(lc, FRK)[r], be = fa(lc, FB)[r];
                const float eg = __expf(gr);
                fa(lc, FCQ)[r] = okr ? p.scale * rq * eg : 0.f;
                fa(lc, FCK)[r] = okr ? rk * __expf(Gl - gr) : 0.f;
                fa(lc, FAKG)[r] = okr ? be * eg * rk : 0.f;
            }
            // the stage's tiles, and the previous chunk's W group done with A diag(beta e^G rk)
            // (warp 14 polls, the four prep warps share the result through a hardware barrier)
            bool ok = true;
            if (warp == 14) {
                ok = warp_wait(sb + L::B_FULL + 8 * s, (lc >> 1) & 1, flag, geo.err, lane);
                if (ok && lc > 0) ok = warp_wait(sb + L::B_MPW, (lc - 1) & 1, flag, geo.err, lane);
            }
            if (!group_and(ok, 1, 128)) break;
            {
                // A diag(beta e^G rk): thread -> row at/2, 32 columns; rows past the end are zero
                const int r = at >> 1, c0 = (at & 1) * 32;
                const bool okr = r < valid;
                const float4 *fk4 = reinterpret_cast<const float4 *>(fa(lc, FAKG) + c0);
                uint4 u[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) u[c] = umma::ld_shared_v4(st + L::ST_A + umma::off(r, c0 + c * 8, 0));
                float fkv[32];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 a = fk4[i];
                    fkv[4 * i] = a.x, fkv[4 * i + 1] = a.y, fkv[4 * i + 2] = a.z, fkv[4 * i + 3] = a.w;
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t w[4] = {u[c].x, u[c].y, u[c].z, u[c].w};
                    uint32_t wk[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 x = Elt<T>::unpack(w[e]);
                        const int i = c * 8 + 2 * e;
                        wk[e] = Elt<T>::pack(okr ? x.x * fkv[i] : 0.f, okr ? x.y * fkv[i + 1] : 0.f);
                    }
                    st_v4(sb + L::AKG + umma::off(r, c0 + c * 8, 0), wk[0], wk[1], wk[2], wk[3]);
                }
            }
            if (valid < C && at >= valid && at < C) {
                // P rows past the end of the sequence belong to other tokens: zero them (P^T dO sums rows)
#pragma unroll
                for (int c = 0; c < 8; ++c) st_v4(st + L::ST_P + umma::off(at, c * 8, 0), 0u, 0u, 0u, 0u);
            }
            umma::fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(sb + L::B_PREP);  // P^T dO and W need only these
            {
                // Q~ = diag(scale rq e^G) Q in place: thread -> row at & 63, key half at >> 6
                const int r = at & 63;
                const float cq = fa(lc, FCQ)[r];
                const uint32_t blk = st + L::ST_Q0 + (at >> 6) * 8192;
                uint4 u[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) u[c] = umma::ld_shared_v4(blk + umma::off(r, c * 8, 0));
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t w[4] = {u[c].x, u[c].y, u[c].z, u[c].w};
                    uint32_t o4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 x = Elt<T>::unpack(w[e]);
                        o4[e] = Elt<T>::pack(x.x * cq, x.y * cq);
                    }
                    st_v4(blk + umma::off(r, c * 8, 0), o4[0], o4[1], o4[2], o4[3]);
                }
            }
            umma::fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(sb + L::B_PREPQ + 8 * (lc & 1));
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ state gradient (256 threads)
        const int sw = warp - 4, q4 = warp & 3, cg = sw >> 2;
        const int d = q4 * 32 + lane;
        constexpr int HW = BV / 2;  // value columns per thread
        const int cb0 = cg * HW;
        const long long st_base = ((long long)n * Hv + j) * DK * DV;
        const long long seg_base = (((long long)n * Hv + j) * nseg + seg) * DK * DV;
        float hS[HW];
#pragma unroll
        for (int i = 0; i < HW; ++i) {
            const int e = v0 + cb0 + i;
            if (p.seg_start)
                hS[i] = p.seg_start[seg_base + (long long)e * DK + d];
            else
                hS[i] = p.dht ? p.dht[st_base + (p.v_first ? (long long)e * DK + d : (long long)d * DV + e)] : 0.f;
        }
        const BoxStore<BV> box{q4, cg, lane};
        const int bx = cb0 & ~63;  // first column of the stored box that holds this warp's columns
        // dh' of step lcn (the gradient after chunk chunk_of(lcn)) into the operand tile, and on to dH'
        auto write_h = [&](int lcn) {
            // (a dDelta-row warp's newer group in flight is this step's dDelta box)
            if (p.dhn) box.free_tile(q4 < 2 && p.ddelta && lcn > 0);
#pragma unroll
            for (int i = 0; i < HW; i += 16) {
                const int col = cb0 + i;
                store_row16<T>(sb + L::H + (col >> 6) * 16384, d, col & 63, hS + i);
            }
            umma::fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(sb + L::B_EPIB);
            if (p.dhn && lcn < nc)
                box.store(&p.tdh, v0 + bx, q4 * 32, (row0 + chunk_of(lcn)) * Hv + j,
                          sb + L::H + (bx >> 6) * 16384 + q4 * 4096);
        };
        write_h(0);
        float glo = 0.f;
        auto fetch_gl = [&](int lc) {
            const int c = chunk_of(lc);
            const int valid = min(C, len - c * C);
            glo = p.g_cs[(tok0 + (long long)c * C + valid - 1) * Hv + j];
        };
        if (nc > 0) fetch_gl(0);
        for (int lc = 0; lc < nc; ++lc) {
            const int c = chunk_of(lc);
            const float egl = __expf(glo);
            if (lc + 1 < nc) fetch_gl(lc + 1);
            bool okw = true;  // every state warp reaches the hardware barriers below, failed or not
            // round A's barrier: polled by warp 5 alone and shared with the other Delta-row warps (4, 8, 9)
            // through a hardware barrier, so that the MMA thread is the only warp polling on its scheduler
            if (q4 < 2) {
                if (warp == 5) okw = warp_wait(sb + L::B_MA, lc & 1, flag, geo.err, lane);
                okw = group_and(okw, 3, 128);
            }
            if (q4 < 2 && okw) {
                // dDelta rows (lanes 0..63): diag(rk e^{Gl-G}) E + P^T dO
                umma::fence_after();
                const int sr = d;
                const float ck = fa(lc, FCK)[sr];
                // the dDelta box stored last step has been read (the dh' box stored since may stay in flight)
                if (p.ddelta) box.free_tile(p.dhn != nullptr);
#pragma unroll
                for (int i = 0; i < HW; i += 16) {
                    float x[16], y[16];
                    umma::ld16(umma::taddr(tmem, q4 * 32, L::T_E + cb0 + i), x);
                    umma::ld16(umma::taddr(tmem, q4 * 32, L::T_P + cb0 + i), y);
                    umma::ld_wait();
                    const int col = cb0 + i;
#pragma unroll
                    for (int u = 0; u < 16; ++u) x[u] = fmaf(ck, x[u], y[u]);
                    store_row16<T>(sb + L::DL + (col >> 6) * 8192, sr, col & 63, x);
                }
                umma::fence_before();
                umma::fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(sb + L::B_EPIA);
                if (p.ddelta)
                    box.store(&p.tdd, v0 + bx, q4 * 32, (row0 + c) * Hv + j, sb + L::DL + (bx >> 6) * 8192 + q4 * 4096);
            }
            // round B's barrier: polled by warp 4, passed on to the other state warps by a hardware barrier
            // (as in the forward chain)
            if (warp == 5 && okw) okw = warp_wait(sb + L::B_MB, lc & 1, flag, geo.err, lane);
            if (!group_and(okw, 2, 256)) break;  // the eight state warps: all go on, or all leave
            umma::fence_after();
#pragma unroll
            for (int i0 = 0; i0 < HW; i0 += 32) {
                float xb[32];
                umma::ld16(umma::taddr(tmem, q4 * 32, L::T_Y + cb0 + i0), xb);
                umma::ld16(umma::taddr(tmem, q4 * 32, L::T_Y + cb0 + i0 + 16), xb + 16);
                umma::ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) hS[i0 + i] = fmaf(egl, hS[i0 + i], xb[i]);
            }
            umma::fence_before();
            write_h(lc + 1);
        }
        if (lane == 0 && (p.dhn || p.ddelta)) tma::wait_all();  // the stored boxes are complete
        if (!*flag && p.seg_end) {
#pragma unroll
            for (int i = 0; i < HW; ++i) p.seg_end[seg_base + (long long)(v0 + cb0 + i) * DK + d] = hS[i];
        } else if (!*flag && p.dh0 && seg == 0) {
#pragma unroll
            for (int i = 0; i < HW; ++i) {
                const int e = v0 + cb0 + i;
                p.dh0[st_base + (p.v_first ? (long long)e * DK + d : (long long)d * DV + e)] = hS[i];
            }
        }
    } else {
        // ------------------------------------------------------------ -W (warps 2, 3; TMEM lanes 64..127)
        const int r = (warp - 2) * 32 + lane;
        const int lb = 32 * (warp & 3);
        for (int lc = 0; lc < nc; ++lc) {
            if (!warp_wait(sb + L::B_MPW, lc & 1, flag, geo.err, lane)) break;
            umma::fence_after();
#pragma unroll
            for (int c = 0; c < 128; c += 64) {
                float x[64];
#pragma unroll
                for (int u = 0; u < 64; u += 16) umma::ld16(umma::taddr(tmem, lb, L::T_W + c + u), x + u);
                umma::ld_wait();
#pragma unroll
                for (int u = 0; u < 64; ++u) x[u] = -x[u];
#pragma unroll
                for (int u = 0; u < 64; u += 16) store_row16<T>(sb + L::WS + (c >> 6) * 8192, r, u, x + u);
            }
            umma::fence_before();
            umma::fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(sb + L::B_EPIA);
        }
    }

    umma::fence_before();
    __syncthreads();
    if (warp == 0) umma::dealloc(tmem, 512);
}

template <typename T, int BV>
__global__ void __launch_bounds__(WS_NT, 1) chain_rev_kernel(Geo geo, const __grid_constant__ RevP p) {
    griddep_launch_next();
    griddep_wait();
    ws_rev_body<T, BV>(geo, p, blockIdx.x, blockIdx.y, blockIdx.z);
}

// The backward's two chains side by side: blocks z < N recompute the forward states (all 128 value
// columns, no output), blocks z >= N run the reverse chain.
template <typename T>
__global__ void __launch_bounds__(WS_NT, 1) chain_ws_pair_kernel(Geo geo, const __grid_constant__ WsP pf,
                                                                 const __grid_constant__ RevP pb) {
    if ((int)blockIdx.z < geo.N)
        ws_fwd_body<T, 128, false>(geo, pf, 0, blockIdx.y, blockIdx.z);
    else
        ws_rev_body<T, 128>(geo, pb, 0, blockIdx.y, blockIdx.z - geo.N);
}

bool ws_map(CUtensorMap *m, const void *base, const Args &a, int heads, int cols) {
    return make_token_map(m, base, a.bf16, cols, heads, (uint64_t)a.B * (uint64_t)a.T, 64);
}

// Per-chunk tiles [rows x Hv][rows_per][128 columns] (states, Delta and their gradients), 64 x 32 boxes.
bool box_map(CUtensorMap *m, void *base, const Args &a, uint64_t rows_per) {
    const uint64_t srows = (uint64_t)a.max_chunks * a.Hv;
    return make_tmap_3d(m, base, a.bf16, DV, rows_per, srows, DV * 2, rows_per * DV * 2, 64, 32, 1);
}

// 64-column slices (two CTAs per chain, the shorter chunk step) unless they would take more waves of one
// CTA per SM than whole-width CTAs do, for batches of equal-length sequences (a packed batch's time is its
// longest sequence's chain, which the shorter step serves better).
template <typename T, int BV>
cudaError_t chain_rev_launch(const Args &a, const RevP &p, int chains, cudaStream_t s) {
    auto kern = chain_rev_kernel<T, BV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, RLay::BYTES);
    if (e != cudaSuccess) return e;
    return launch_overlapped(kern, dim3(DV / BV, a.Hv, chains), dim3(WS_NT), RLay::BYTES, s, make_geo(a), p);
}

template <typename T>
cudaError_t chain_rev_t(const Args &a, const RevP &p, cudaStream_t s) {
    const int chains = a.N * (p.nseg > 1 ? p.nseg : 1);
    int dev = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const long long ctas = (long long)chains * a.Hv;
    const bool wide = a.cu == nullptr && sms > 0 && (2 * ctas + sms - 1) / sms > (ctas + sms - 1) / sms;
    return wide ? chain_rev_launch<T, 128>(a, p, chains, s) : chain_rev_launch<T, 64>(a, p, chains, s);
}

template <typename T, int BV, bool WRITE_O>
cudaError_t chain_ws_t(const Args &a, const WsP &p, cudaStream_t s) {
    auto kern = chain_ws_kernel<T, BV, WRITE_O>;
    const uint32_t bytes = Lay<BV, WRITE_O>::BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    return launch_overlapped(kern, dim3(DV / BV, a.Hv, a.N * (p.nseg > 1 ? p.nseg : 1)), dim3(WS_NT), bytes, s,
                             make_geo(a), p);
}

template <typename T>
cudaError_t chain_ws_pair_t(const Args &a, const WsP &pf, const RevP &pb, cudaStream_t s) {
    auto kern = chain_ws_pair_kernel<T>;
    const uint32_t bytes = Lay<128, false>::BYTES > RLay::BYTES ? Lay<128, false>::BYTES : RLay::BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    return launch_plain(kern, dim3(1, a.Hv, 2 * a.N), dim3(WS_NT), bytes, s, make_geo(a), pf, pb);
}

}  // namespace

cudaError_t launch_chain_ws_pair(const Args &a, const void *q, const void *k, const void *v, const float *g_cs,
                                 const void *beta, const void *A, const void *P, const float *rq, const float *rk,
                                 const float *h0, void *h, void *delta, const void *dout, const float *dht,
                                 void *dhn, void *ddelta, float *dh0, cudaStream_t s) {
    WsP pf;
    RevP pb;
    if (!ws_map(&pf.tq, q, a, a.Hq, a.K) || !ws_map(&pf.tk, k, a, a.Hq, a.K) || !ws_map(&pf.tv, v, a, a.Hv, a.V) ||
        !ws_map(&pf.ta, A, a, a.Hv, C) || !ws_map(&pb.tq, q, a, a.Hq, a.K) || !ws_map(&pb.tk, k, a, a.Hq, a.K) ||
        !ws_map(&pb.tdo, dout, a, a.Hv, a.V) || !ws_map(&pb.tp, P, a, a.Hv, C) || !ws_map(&pb.ta, A, a, a.Hv, C))
        return cudaErrorInvalidValue;
    pf.tp = pb.tp;
    pf.tma_h = h != nullptr;
    pf.tma_delta = delta != nullptr;
    if ((h && !box_map(&pf.th, h, a, DK)) || (delta && !box_map(&pf.tdl, delta, a, C)) ||
        (dhn && !box_map(&pb.tdh, dhn, a, DK)) || (ddelta && !box_map(&pb.tdd, ddelta, a, C)))
        return cudaErrorInvalidValue;
    pf.g_cs = g_cs;
    pf.h0 = h0;
    pf.rq = rq;
    pf.rk = rk;
    pf.beta = beta;
    pf.o = nullptr;
    pf.fin = nullptr;
    pf.h = h;
    pf.delta = delta;
    pf.seg_start = nullptr;
    pf.nseg = 1;
    pf.affine = false;
    pf.gate_f32 = a.gate_f32;
    pf.l2norm = a.l2norm;
    pf.v_first = a.v_first;
    pf.h_vfirst = false;
    pf.scale = a.scale;
    pb.g_cs = g_cs;
    pb.rq = rq;
    pb.rk = rk;
    pb.dht = dht;
    pb.seg_start = nullptr;
    pb.nseg = 1;
    pb.seg_end = nullptr;
    pb.beta = beta;
    pb.dhn = dhn;
    pb.ddelta = ddelta;
    pb.dh0 = dh0;
    pb.gate_f32 = a.gate_f32;
    pb.l2norm = a.l2norm;
    pb.v_first = a.v_first;
    pb.scale = a.scale;
    return a.bf16 ? chain_ws_pair_t<__nv_bfloat16>(a, pf, pb, s) : chain_ws_pair_t<__half>(a, pf, pb, s);
}

cudaError_t launch_chain_rev(const Args &a, const void *q, const void *k, const float *g_cs, const void *beta,
                             const void *A, const void *P, const float *rq, const float *rk, const void *dout,
                             const float *dht, const float *seg_start, int nseg, void *dhn, void *ddelta, float *dh0,
                             float *seg_end, cudaStream_t s) {
    RevP pb;
    if (!ws_map(&pb.tq, q, a, a.Hq, a.K) || !ws_map(&pb.tk, k, a, a.Hq, a.K) || !ws_map(&pb.tdo, dout, a, a.Hv, a.V) ||
        !ws_map(&pb.tp, P, a, a.Hv, C) || !ws_map(&pb.ta, A, a, a.Hv, C) ||
        (dhn && !box_map(&pb.tdh, dhn, a, DK)) || (ddelta && !box_map(&pb.tdd, ddelta, a, C)))
        return cudaErrorInvalidValue;
    pb.g_cs = g_cs;
    pb.rq = rq;
    pb.rk = rk;
    pb.dht = dht;
    pb.seg_start = seg_start;
    pb.nseg = nseg;
    pb.seg_end = seg_end;
    pb.beta = beta;
    pb.dhn = dhn;
    pb.ddelta = ddelta;
    pb.dh0 = dh0;
    pb.gate_f32 = a.gate_f32;
    pb.l2norm = a.l2norm;
    pb.v_first = a.v_first;
    pb.scale = a.scale;
    return a.bf16 ? chain_rev_t<__nv_bfloat16>(a, pb, s) : chain_rev_t<__half>(a, pb, s);
}

cudaError_t launch_chain_ws(const Args &a, const void *q, const void *k, const void *v, const float *g_cs,
                            const void *beta, const void *A, const void *P, const float *rq, const float *rk,
                            const float *h0, const float *seg_start, int nseg, void *o, float *final_state, void *h,
                            bool h_vfirst, void *delta, cudaStream_t s) {
    WsP p;
    const uint64_t tokens = (uint64_t)a.B * (uint64_t)a.T;
    if (!ws_map(&p.tq, q, a, a.Hq, a.K) || !ws_map(&p.tk, k, a, a.Hq, a.K) || !ws_map(&p.tv, v, a, a.Hv, a.V) ||
        !ws_map(&p.ta, A, a, a.Hv, C) || (o && !ws_map(&p.tp, P, a, a.Hv, C)) ||
        (o && !make_token_map(&p.to, o, a.bf16, a.V, a.Hv, tokens, 32)))
        return cudaErrorInvalidValue;
    p.g_cs = g_cs;
    p.rq = rq;
    p.rk = rk;
    p.h0 = h0;
    p.beta = beta;
    p.o = o;
    p.fin = final_state;
    p.h = h;
    p.delta = delta;
    p.seg_start = seg_start;
    p.nseg = nseg;
    p.affine = false;
    p.gate_f32 = a.gate_f32;
    p.l2norm = a.l2norm;
    p.v_first = a.v_first;
    p.h_vfirst = h_vfirst;
    p.scale = a.scale;
    // the states leave as TMA boxes (the [K][V] layout; the [V][K] layout by direct stores), Delta likewise
    p.tma_h = h != nullptr && !h_vfirst;
    p.tma_delta = delta != nullptr;
    if ((p.tma_h && !box_map(&p.th, h, a, DK)) || (p.tma_delta && !box_map(&p.tdl, delta, a, C)))
        return cudaErrorInvalidValue;
    if (o)
        return a.bf16 ? chain_ws_t<__nv_bfloat16, 64, true>(a, p, s) : chain_ws_t<__half, 64, true>(a, p, s);
    return a.bf16 ? chain_ws_t<__nv_bfloat16, 64, false>(a, p, s) : chain_ws_t<__half, 64, false>(a, p, s);
}

cudaError_t launch_chain_ws_affine(const Args &a, const void *q, const void *k, const void *v, const float *g_cs,
                                   const void *beta, const void *A, const float *rq, const float *rk, int nseg,
                                   float *end0, float *end1, cudaStream_t s) {
    WsP p;
    if (nseg < 2 || !ws_map(&p.tq, q, a, a.Hq, a.K) || !ws_map(&p.tk, k, a, a.Hq, a.K) ||
        !ws_map(&p.tv, v, a, a.Hv, a.V) || !ws_map(&p.ta, A, a, a.Hv, C))
        return cudaErrorInvalidValue;
    p.g_cs = g_cs;
    p.rq = rq;
    p.rk = rk;
    p.h0 = nullptr;
    p.beta = beta;
    p.o = nullptr;
    p.fin = nullptr;
    p.h = nullptr;
    p.delta = nullptr;
    p.seg_start = nullptr;
    p.nseg = nseg;
    p.affine = true;
    p.seg_end[0] = end0;
    p.seg_end[1] = end1;
    p.gate_f32 = a.gate_f32;
    p.l2norm = a.l2norm;
    p.v_first = a.v_first;
    p.h_vfirst = false;
    p.scale = a.scale;
    p.tma_h = false;
    p.tma_delta = false;
    auto kern = a.bf16 ? chain_ws_kernel<__nv_bfloat16, 128, false> : chain_ws_kernel<__half, 128, false>;
    const uint32_t bytes = Lay<128, false>::BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    // block x: the kind (the slice is the whole width)
    return launch_overlapped(kern, dim3(2, a.Hv, a.N * nseg), dim3(WS_NT), bytes, s, make_geo(a), p);
}

}  // namespace gdr
