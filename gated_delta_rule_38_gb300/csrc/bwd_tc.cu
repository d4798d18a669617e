// Per-chunk gradients of the chunked gated delta rule on tcgen05, and the
// sequence-level gate-gradient pass.
//
// bwd_chunk_tc: one persistent CTA of 512 threads per SM walks (chunk, q/k head)
// items, visiting the value heads of each item's group in order.  Tokens are the
// rows of every product.  Two 64-row operands that share their B operand are
// stacked into one M=128 MMA, so TMEM lanes 0..63 hold one result and lanes
// 64..127 the other; dq rows accumulate in the registers of the lane-0..63
// threads and dk rows in those of the lane-64..127 threads (each thread holds a
// quarter of a row).  dq is stored after round 3 of the item's last head, dk
// after round 5.  With h the state before
// the chunk, dH' the gradient after it, Delta and dDelta from the two chains:
//
//   round 1: [dO;dDelta] h^T        -> dq += scale e^{G} dO h^T ;  dW = -dDelta h^T
//            [V;Delta] dH'^T        -> dk += e^{Gl-G} Delta dH'^T
//            [dO;dDelta] [V;Delta]^T-> dP = dO Delta^T (-> dS = scale dP o Gamma o M), dA2 = dDelta V^T
//            [Q;K] K^T              -> KK^T
//   round 2: [A^T;A^T] [dDelta | dW]  -> dv = beta A^T dDelta, A^T dW (dbeta), dk += diag(beta e^G) A^T dW
//            dW K^T                 -> dA = (dW K^T diag(e^G) + dDelta V^T) diag(beta), strictly lower
//   round 3: dA A^T -> X ;  dq += dS K ;  dk += dS^T Q
//   round 4: dL = -A^T X ;  dKK = dL o beta_r Gamma  ;  dbeta += sum_s dL Gamma KK
//   round 5: dk += dKK K + dKK^T K
//
// dbeta_r = e^{G_r} <(A^T dW)_r, k_r> + <(A^T dDelta)_r, v_r> + sum_s dL_rs Gamma_rs KK_rs.
// dG_r (gradient w.r.t. the chunk-local cumsum G) collects the decay terms of P (E = dP o P)
// and L (F = dL o L) as row sums minus column sums, <q_r, scale e^{G_r} (dO h^T)_r>,
// -e^{Gl-G_r} <(Delta dH'^T)_r, k_r>, beta_r e^{G_r} <(A^T dW)_r, k_r>, and at the last valid
// row e^{Gl} <dH', h> plus the sum of the key terms; dg is its reverse cumsum inside the chunk.
// All reductions run in a fixed order (deterministic results).
#include <cuda_runtime.h>

#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tmap.h"
#include "umma.cuh"

namespace gdr {
namespace {

constexpr int NT = 512;
// ---- shared memory (bytes from a 1024-aligned base)
constexpr uint32_t S_Q0 = 0, S_K0 = 8192;             // [Q b0][K b0][Q b1][K b1]
constexpr uint32_t S_DO0 = 32768, S_DD0 = 40960;      // [dO b0][dDelta b0][dO b1][dDelta b1]
constexpr uint32_t S_X = 65536, S_DW0 = 73728, S_DS = 81920, S_DW1 = 90112;
constexpr uint32_t S_V0 = 98304, S_D0 = 106496;       // [V b0][Delta b0][V b1][Delta b1]
constexpr uint32_t S_DA = S_D0, S_DKK = S_D0 + 16384; // reuse Delta's blocks after round 1
constexpr uint32_t S_H = 131072, S_DH = 163840;       // [128 x 64] blocks of 16 KB
constexpr uint32_t S_A = 196608, S_A2 = 204800;   // A, and a second copy of it (the stacked round-2 operand)
constexpr uint32_t S_F = 212992;                      // scalars
constexpr uint32_t S_BAR = S_F + 52 * 64 * 4, S_LBAR = S_BAR + 8, S_SLOT = S_LBAR + 8, S_FLAG = S_SLOT + 4,
                   S_USED = S_FLAG + 4;
constexpr uint32_t S_BYTES = S_USED + 1024;
// scalar slots (64 floats each)
// (per column quarter q of a row: slot + q; column sums per row half: slot + 0/1)
enum {
    F_G = 0, F_B, F_EG, F_EL, F_QD0, F_VD0 = F_QD0 + 4, F_KD0 = F_VD0 + 4, F_LB0 = F_KD0 + 4, F_ER0 = F_LB0 + 4,
    F_EC0 = F_ER0 + 4, F_Z0 = F_EC0 + 2, F_FR0 = F_Z0 + 4, F_FC0 = F_FR0 + 4, F_HD = F_FC0 + 2, F_DG, F_IQ, F_IK,
    F_MQ, F_MK, F_PDG, F_PDB, F_DP, F_COUNT = F_DP + 8
};
// TMEM columns
constexpr uint32_t T_R1 = 0, T_R2 = 128, T_R3 = 256, T_R4 = 384, T_R8 = 448, T_COLS = 512;

template <typename T> struct IsBf16 { static constexpr bool value = false; };
template <> struct IsBf16<__nv_bfloat16> { static constexpr bool value = true; };

struct BcP {
    // TMA maps: q, k [tokens][Hq][K]; dO, v [tokens][Hv][V]; A [tokens][Hv][64];
    // states h, dH' [rows*Hv][128][128]; Delta, dDelta [rows*Hv][64][128]
    // outputs dq, dk [tokens][Hq][K], dv [tokens][Hv][V] (full chunks leave by TMA stores)
    // (K, V below 128: the 128-wide tiles load zeros past them and the stores are clipped)
    CUtensorMap tq, tk, tdo, tv, ta, th, tdh, td, tdd, tdq, tdk, tdv;
    const void *q, *k, *v, *A, *beta, *dout, *h, *dhn, *delta, *ddelta;
    const float *g_cs;
    void *dq, *dk, *dv, *dg, *dbeta;
    bool gate_f32, l2norm;
    float scale;
    int nslots;  // chunk slots (dense: B * ceil(T/64); varlen: the chunk-table bound)
};

// Column sums of a 32 x 16 block held one row per lane (v[c] = column c): lane l ends with the sum over
// the 32 lanes of column l & 15 (fixed-order butterfly, 16 shuffles).
__device__ __forceinline__ float colsum16(float (&v)[16], int lane) {
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float send = up ? v[i] : v[i + o];
            const float keep = up ? v[i + o] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 16);
}

template <typename T>
__device__ __forceinline__ void store16(uint32_t base, int row, int col0, const float *x) {
#pragma unroll
    for (int c = 0; c < 2; ++c)
        umma::st_shared_v4(base + umma::off(row, col0 + c * 8, 0), Elt<T>::pack(x[c * 8], x[c * 8 + 1]),
                           Elt<T>::pack(x[c * 8 + 2], x[c * 8 + 3]), Elt<T>::pack(x[c * 8 + 4], x[c * 8 + 5]),
                           Elt<T>::pack(x[c * 8 + 6], x[c * 8 + 7]));
}

// 16 values of row `row`, columns col0.. of a swizzled tile, as floats.
template <typename T>
__device__ __forceinline__ void load16(uint32_t base, int row, int col0, float *x) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const uint4 u = umma::ld_shared_v4(base + umma::off(row, col0 + c * 8, 0));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = Elt<T>::unpack(w[e]);
            x[c * 8 + 2 * e] = f.x;
            x[c * 8 + 2 * e + 1] = f.y;
        }
    }
}

// A gate element's raw bits (bf16 / fp16 in the low half) as a float.
template <typename T> __device__ __forceinline__ float bits_to_f(uint32_t b);
template <> __device__ __forceinline__ float bits_to_f<__nv_bfloat16>(uint32_t b) { return __uint_as_float(b << 16); }
template <> __device__ __forceinline__ float bits_to_f<__half>(uint32_t b) {
    return __half2float(__ushort_as_half((unsigned short)b));
}

// Row norms of the 64 rows of a [64 x 128] swizzled tile (blocks 16 KB apart), read only: eight warps per tile,
// four lanes per row; lane quarter qq takes 16-byte chunks 2qq, 2qq+1 of each 64-column block, so the eight
// lanes of a quarter-warp access hit eight distinct bank groups.  n_out[r] = 1 / sqrt(|x_r|^2 + eps) (the
// factor that normalises the row), m_out[r] = sqrt(|x_r|^2 + eps).
template <typename T>
__device__ __forceinline__ void row_norms64(uint32_t base, int warp, int lane, float *n_out, float *m_out) {
    const int rq = lane >> 2, qq = lane & 3;
    const int r = warp * 8 + rq;  // warps 0..7 x 8 rows
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint4 u = umma::ld_shared_v4(base + (uint32_t)(c >> 1) * 16384u + umma::off(r, (qq * 2 + (c & 1)) * 8, 0));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 x = Elt<T>::unpack(w[e]);
            ss += x.x * x.x + x.y * x.y;
        }
    }
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    if (qq == 0) {
        const float m = sqrtf(ss + L2_EPS);
        n_out[r] = 1.0f / m;
        m_out[r] = m;
    }
}

template <typename T>
__global__ void __launch_bounds__(NT, 1) bwd_chunk_tc_kernel(Geo geo, const __grid_constant__ BcP p) {
    griddep_launch_next();
    griddep_wait();
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const int Hv = geo.Hv, Hq = geo.Hq, grp = Hv / Hq;
    // Persistent: this CTA walks the work items w = blockIdx.x, + gridDim.x, ... (item = chunk slot x q/k
    // head, each with the grp value heads of its group: one "unit" per value head).  The tiles of the next
    // unit are prefetched into buffers as soon as the current unit is done with them.
    // (32-bit item arithmetic: the host keeps chunk slots x Hq below 2^31)
    const int nitems = p.nslots * Hq;
    auto next_item = [&](int w_) -> int {
        for (; w_ < nitems; w_ += (int)gridDim.x)
            if (geo.has_chunk(geo.div_hq(w_))) return w_;
        return -1;
    };
    // a unit's place: first token t, valid rows, q/k head, value head, state row (chunk row x Hv + value head)
    struct Pos {
        int t, valid, hq, j, row;
    };
    auto locate = [&](int w_, int jj_) {
        Pos u;
        const int slot_ = geo.div_hq(w_);
        long long t_;
        int n_, c_;
        geo.chunk(slot_, t_, u.valid, n_, c_);
        u.t = (int)t_;
        u.hq = w_ - slot_ * Hq;
        u.j = u.hq * grp + jj_;
        u.row = slot_ * Hv + u.j;
        return u;
    };
    int wit = next_item(blockIdx.x);
    if (wit < 0) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L = (warp & 3) * 32 + lane, qc = warp >> 2, lb = (warp & 3) * 32;  // qc: column quarter
    const bool upper = L >= 64;
    const int uw = (warp >> 2) * 2 + (warp & 1);  // index of this warp among the upper (or lower) eight
    const int r = L & 63;  // token row of this thread's TMEM lane
    constexpr bool bf16 = IsBf16<T>::value;
    float *F = reinterpret_cast<float *>(smem + S_F);
    auto f = [&](int slot_, int i) -> float & { return F[slot_ * 64 + i]; };
    const uint32_t bar = sb + S_BAR;
    volatile int *sflag = reinterpret_cast<volatile int *>(smem + S_FLAG);

    const uint32_t lbar = sb + S_LBAR;  // tile loads
    if (tid == 0) {
        umma::mbar_init(bar, 1);
        umma::mbar_init(lbar, 1);
        umma::fence_mbar_init();
        *sflag = 0;
    }
    if (warp == 0) umma::alloc(sb + S_SLOT, T_COLS);
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + S_SLOT);

    // instruction descriptors
    const uint32_t i_n128 = umma::idesc(128, 128, bf16, false, false);
    const uint32_t i_n64 = umma::idesc(128, 64, bf16, false, false);
    const uint32_t i_n256_mn = umma::idesc(128, 256, bf16, true, true);
    const uint32_t i_n128_bmn = umma::idesc(128, 128, bf16, false, true);
    const uint32_t i_n128_mn = umma::idesc(128, 128, bf16, true, true);
    const uint32_t i_n64_mn = umma::idesc(128, 64, bf16, true, true);
    // operand descriptors (K-major: sbo 1024; MN-major: lbo = distance between 64-wide blocks)
    const uint64_t dDOa = umma::desc(sb + S_DO0, 16, 1024);         // [dO; dDelta] rows, K = value
    const uint64_t dH = umma::desc(sb + S_H, 16, 1024);             // h[d][e]: n = d, k = e
    const uint64_t dVa = umma::desc(sb + S_V0, 16, 1024);           // [V; Delta] rows, K = value
    const uint64_t dDH = umma::desc(sb + S_DH, 16, 1024);           // dH'[d][e]
    const uint64_t dQa = umma::desc(sb + S_Q0, 16, 1024);           // [Q; K] rows, K = key
    const uint64_t dKa = umma::desc(sb + S_K0, 16, 1024);           // K rows (n = token), K = key
    const uint64_t dAmn = umma::desc(sb + S_A, 8192, 1024);         // [A^T; A^T] (m = row), k = token
    const uint64_t dDDmn = umma::desc(sb + S_DD0, 16384, 1024);     // [dDelta | dW] (n = col), k = token
    const uint64_t dWup = umma::desc(sb + S_DW0 - 8192, 16, 1024);  // rows 64..127 = dW, K = key
    const uint64_t dDA = umma::desc(sb + S_DA, 16, 1024);           // dA rows, K = token
    const uint64_t dAk = umma::desc(sb + S_A, 16, 1024);            // A rows as K-major B (n = token)
    const uint64_t dDS = umma::desc(sb + S_DS, 16, 1024);           // dS rows (lanes 0..63)
    const uint64_t dKmn = umma::desc(sb + S_K0, 16384, 1024);       // K (n = key col), k = token
    const uint64_t dQmn = umma::desc(sb + S_Q0, 16384, 1024);       // Q (n = key col), k = token
    const uint64_t dDSup = umma::desc(sb + S_DS - 8192, 8192, 1024);  // m 64..127 = dS^T
    const uint64_t dAup = umma::desc(sb + S_A - 8192, 8192, 1024);    // m 64..127 = A^T
    const uint64_t dXmn = umma::desc(sb + S_X, 8192, 1024);           // X (n = col), k = token
    const uint64_t dKKk = umma::desc(sb + S_DKK - 8192, 16, 1024);    // rows 64..127 = dKK
    const uint64_t dKKmn = umma::desc(sb + S_DKK - 8192, 8192, 1024); // m 64..127 = dKK^T

    uint32_t phase = 0, lphase = 0;
    auto wait_mma = [&]() -> bool {
        if (tid == 0 && !umma::mbar_spin(bar, phase)) {
            raise_error(geo.err, GDR_ERR_TIMEOUT);
            *sflag = 1;
        }
        phase ^= 1;
        umma::fence_before();
        __syncthreads();
        umma::fence_after();
        return *sflag == 0;
    };
    auto sync_tc = [&]() {
        umma::fence_async_smem();
        umma::fence_before();
        __syncthreads();
        umma::fence_after();
    };

    float acc[32];  // dq row (lower lanes) or dk row (upper lanes), key columns 32*qc..
    bool ok = true;

    // tile loads of unit u (value head jj_ of its item's group), in groups by the point where the current
    // unit frees the buffers: 1 = h, dH', dO (after round 1, beside round 2); 2 = V, dDelta (after round 3 is issued);
    // 3 = Delta's first column block (the dA block, after round 4 is issued); 4 = A (after round 5 is
    // issued); 5 = q for the first head of an item (after dq is stored); 6 = k for the first head of an item
    // and Delta's second column block (the dKK block, after the unit).  All bytes of a unit are announced on
    // the load barrier with its first group.
    auto unit_bytes = [&](int jj_) -> uint32_t { return 32768u * 2 + 16384u + 16384u * 2 + 16384u + 8192u * 2 +
                                                         (jj_ == 0 ? 32768u : 0u); };
    auto issue = [&](const Pos &u, int jj_, int group) {
        const int t = u.t, row = u.row, j_ = u.j, hq_ = u.hq;
        if (group == 1) {
            tma::expect_tx(lbar, unit_bytes(jj_));
            tma::load3d(sb + S_H, &p.th, 0, 0, row, lbar);
            tma::load3d(sb + S_H + 16384, &p.th, 64, 0, row, lbar);
            tma::load3d(sb + S_DH, &p.tdh, 0, 0, row, lbar);
            tma::load3d(sb + S_DH + 16384, &p.tdh, 64, 0, row, lbar);
            tma::load3d(sb + S_DO0, &p.tdo, 0, j_, t, lbar);
            tma::load3d(sb + S_DO0 + 16384, &p.tdo, 64, j_, t, lbar);
        } else if (group == 2) {
            tma::load3d(sb + S_V0, &p.tv, 0, j_, t, lbar);
            tma::load3d(sb + S_V0 + 16384, &p.tv, 64, j_, t, lbar);
            tma::load3d(sb + S_DD0, &p.tdd, 0, 0, row, lbar);
            tma::load3d(sb + S_DD0 + 16384, &p.tdd, 64, 0, row, lbar);
        } else if (group == 3) {
            tma::load3d(sb + S_D0, &p.td, 0, 0, row, lbar);
        } else if (group == 4) {
            tma::load3d(sb + S_A, &p.ta, 0, j_, t, lbar);
            tma::load3d(sb + S_A2, &p.ta, 0, j_, t, lbar);
        } else if (group == 5) {
            if (jj_ == 0) {
                tma::load3d(sb + S_Q0, &p.tq, 0, hq_, t, lbar);
                tma::load3d(sb + S_Q0 + 16384, &p.tq, 64, hq_, t, lbar);
            }
        } else {
            tma::load3d(sb + S_D0 + 16384, &p.td, 64, 0, row, lbar);
            if (jj_ == 0) {
                tma::load3d(sb + S_K0, &p.tk, 0, hq_, t, lbar);
                tma::load3d(sb + S_K0 + 16384, &p.tk, 64, hq_, t, lbar);
            }
        }
    };
    // gates of a unit (threads GT..GT+63), fetched one unit ahead as raw loads that are converted only at the
    // next unit's top, so no thread waits for them in the middle of a unit
    constexpr int GT = 64;
    // (each value is written by its own predicated load and read by nothing before that point)
    float gnext = 0.f, bnext32 = 0.f;
    uint32_t bnext16 = 0u;
    auto fetch_gates = [&](const Pos &u) {
        const int i = tid - GT, v_ = u.valid;
        if (i >= 0 && i < C) {
            const long long ti = ((long long)u.t + i) * Hv + u.j;
            gnext = 0.f;
            bnext32 = 0.f;
            bnext16 = 0u;
            if (i < v_) gnext = p.g_cs[ti];
            if (i < v_ && p.gate_f32) bnext32 = static_cast<const float *>(p.beta)[ti];
            if (i < v_ && !p.gate_f32) bnext16 = static_cast<const unsigned short *>(p.beta)[ti];
        }
    };
    // the tile loads of groups 1 and 6 are issued by thread TT (an upper-lane thread, whose epilogues are the
    // lighter ones), those of groups 2, 3 and 4 by the MMA thread right after it has issued rounds 3, 4 and 5,
    // and group 5 by thread ST once dq has left
    constexpr int TT = 64;
    // Full chunks (64 valid rows) leave through shared memory: the rows are written into freed operand blocks in
    // the tile layout and thread ST (a lower-lane thread) stores them with TMA; a ragged chunk's rows are stored
    // directly (its tail rows belong to the next sequence).  Staging blocks: dv -> dW's (after round 2),
    // dq -> X and dW0 (after round 4), dk -> dS and dW1 (after round 5).  ST waits for its stores to finish
    // reading before a barrier that precedes the next writes to those blocks.
    constexpr int ST = 32;
    // dq (lower lanes) / dk (upper lanes) rows, straight from the registers: with x the raw row (the q or k tile
    // in shared memory), n = 1 / sqrt(|x|^2 + eps) and xh = n x, dx = (dxh - xh (xh . dxh)) n
    // = (dxh - x n^2 (x . dxh)) n; the four column quarters of a row meet through one partial dot product each
    const uint32_t xt = sb + (upper ? S_K0 : S_Q0) + (qc >> 1) * 16384;
    const int xc = (qc & 1) * 32;  // this thread's key columns within the 64-column block
    float *dp = &f(F_DP, 0);       // [4 quarters][128 lanes]
    auto dot_partial = [&]() {
        float part = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint4 u = umma::ld_shared_v4(xt + umma::off(r, xc + c * 8, 0));
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 x = Elt<T>::unpack(w[e]);
                part = fmaf(x.x, acc[c * 8 + 2 * e], fmaf(x.y, acc[c * 8 + 2 * e + 1], part));
            }
        }
        dp[qc * 128 + L] = part;
    };
    auto store_row = [&](long long tok0_, int valid_, int hq_) {
        const bool staged = valid_ == C;
        if (!staged && r >= valid_) return;
        const float inv = p.l2norm ? f(upper ? F_IK : F_IQ, r) : 1.f;
        const float dot = p.l2norm ? inv * inv * ((dp[L] + dp[128 + L]) + (dp[256 + L] + dp[384 + L])) : 0.f;
        T *dst = static_cast<T *>(upper ? p.dk : p.dq) + ((tok0_ + r) * Hq + hq_) * geo.K + qc * 32;
        const uint32_t stg = sb + (upper ? ((qc >> 1) ? S_DW1 : S_DS) : ((qc >> 1) ? S_DW0 : S_X));
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float xv[8];
            if (p.l2norm) {
                const uint4 u = umma::ld_shared_v4(xt + umma::off(r, xc + c * 8, 0));
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 x = Elt<T>::unpack(w[e]);
                    xv[2 * e] = x.x;
                    xv[2 * e + 1] = x.y;
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) xv[e] = 0.f;
            }
            uint32_t o4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                o4[e] = Elt<T>::pack((acc[c * 8 + 2 * e] - xv[2 * e] * dot) * inv,
                                     (acc[c * 8 + 2 * e + 1] - xv[2 * e + 1] * dot) * inv);
            if (staged)
                umma::st_shared_v4(stg + umma::off(r, xc + c * 8, 0), o4[0], o4[1], o4[2], o4[3]);
            else if (qc * 32 + c * 8 < geo.K)
                *reinterpret_cast<uint4 *>(dst + c * 8) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
        }
    };

    int jj = 0;
    bool posted = false;  // a unit's loads are announced and not yet waited for
    Pos cur = locate(wit, 0);
    if (tid == TT)
        for (int g = 1; g <= 6; ++g) issue(cur, 0, g);
    posted = true;
    fetch_gates(cur);

    while (ok) {
        const long long tok0 = cur.t;
        const int valid = cur.valid, hq = cur.hq, j = cur.j;
        const bool last_head = jj + 1 == grp;  // dq and dk of the item are complete in this unit
        // the unit after this one, located once here (while the tiles are still on their way)
        int wn = wit;
        int jn = jj + 1;
        if (jn == grp) {
            jn = 0;
            wn = next_item(wit + (int)gridDim.x);
        }
        Pos nxt = cur;
        if (wn >= 0) nxt = locate(wn, jn);
        if (jj == 0) {
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = 0.f;
        }
        if (tid >= GT && tid < GT + C) {
            f(F_G, tid - GT) = gnext;
            f(F_B, tid - GT) = p.gate_f32 ? bnext32 : bits_to_f<T>(bnext16);
        }
        if (tid == 0 && !umma::mbar_spin(lbar, lphase)) {  // the barrier below passes it on
            raise_error(geo.err, GDR_ERR_TIMEOUT);
            *sflag = 1;
        }
        lphase ^= 1u;
        posted = false;
        if (tid == ST) tma::wait_read();  // the previous unit's dq / dk staging blocks are free again
        umma::fence_before();
        __syncthreads();
        umma::fence_after();
        if (*sflag) {
            ok = false;
            break;
        }

        // ---------------- round 1 (raw q and k tiles: the L2 normalisation enters every product that uses
        //                  them as a per-row or per-column factor, so nothing has to be rewritten first)
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t ko = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
                umma::mma(tmem + T_R1, dDOa + ko, dH + ko, i_n128, ks > 0);
                umma::mma(tmem + T_R2, dVa + ko, dDH + ko, i_n128, ks > 0);
                umma::mma(tmem + T_R3, dDOa + ko, dVa + ko, i_n128, ks > 0);
                umma::mma(tmem + T_R4, dQa + ko, dKa + ko, i_n64, ks > 0);
            }
            umma::commit(bar);
        }
        // while round 1 runs: decays, and the q / k row norms of a new item (warps 0..7 q, 8..15 k)
        const float Gl = f(F_G, valid - 1);
        if (tid < C) {
            f(F_EG, tid) = __expf(f(F_G, tid));
            f(F_EL, tid) = __expf(Gl - f(F_G, tid));
        }
        if (jj == 0) {
            if (p.l2norm) {
                row_norms64<T>(sb + (warp < 8 ? S_Q0 : S_K0), warp & 7, lane, &f(warp < 8 ? F_IQ : F_IK, 0),
                               &f(warp < 8 ? F_MQ : F_MK, 0));
            } else if (tid < 4 * C) {
                f(F_IQ + (tid >> 6), tid & 63) = 1.f;  // F_IQ, F_IK, F_MQ, F_MK
            }
        }
        if (upper) {
            // <dH', h> over the whole state (both tiles share one layout, so equal offsets hold equal elements),
            // on the upper-lane warps while round 1 runs (it reads only the loaded tiles); consecutive threads
            // read consecutive 8-byte words (no bank conflicts)
            const int ut = uw * 32 + lane;
            float hd = 0.f;
#pragma unroll 4
            for (int u = 0; u < (DK * DV * 2 / 8) / (NT / 2); ++u) {
                const uint32_t o = (uint32_t)(u * (NT / 2) + ut) * 8u;
                const uint2 a = *reinterpret_cast<const uint2 *>(smem + S_H + o);
                const uint2 b = *reinterpret_cast<const uint2 *>(smem + S_DH + o);
                const float2 a0 = Elt<T>::unpack(a.x), a1 = Elt<T>::unpack(a.y);
                const float2 b0 = Elt<T>::unpack(b.x), b1 = Elt<T>::unpack(b.y);
                hd += a0.x * b0.x + a0.y * b0.y + a1.x * b1.x + a1.y * b1.y;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) hd += __shfl_xor_sync(0xffffffffu, hd, o);
            if (lane == 0) f(F_HD, uw) = hd;
        }
        if (!wait_mma()) {
            ok = false;
            break;
        }
        if (!upper) {
            float qd = 0.f;  // <q_r, dq_r> of this value head (this thread's quarter of the row)
            const float sc = p.scale * f(F_EG, r);
#pragma unroll
            for (int c = 0; c < 32; c += 16) {
                float x[16], qv[16];
                umma::ld16(umma::taddr(tmem, lb, T_R1 + qc * 32 + c), x);
                load16<T>(sb + S_Q0 + (qc >> 1) * 16384, r, (qc & 1) * 32 + c, qv);
                umma::ld_wait();
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    x[u] *= sc;
                    acc[c + u] += x[u];
                    qd += qv[u] * x[u];
                }
            }
            const float nqr = f(F_IQ, r);
            f(F_QD0 + qc, r) = qd * nqr;  // <q^_r, .> with q^ = nq q
            // dS = scale dP o Gamma o M  (dP = dO Delta^T in columns 64..127 of R3), stored as
            // dS'' = diag(nq) dS diag(nk) for the raw-tile products of round 3;
            // E = dS o (Q^ K^^T) = dS'' o (Q K^T) gives the decay terms of dG (row sums minus column sums)
            const float gr = f(F_G, r);
            float ev[16], er = 0.f;
            {
                const int c = 0;
                float x[16], qk[16];
                umma::ld16(umma::taddr(tmem, lb, T_R3 + 64 + qc * 16), x);
                umma::ld16(umma::taddr(tmem, lb, T_R4 + qc * 16), qk);
                umma::ld_wait();
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int s = qc * 16 + u;
                    x[u] = (s <= r && r < valid) ? p.scale * x[u] * __expf(gr - f(F_G, s)) * nqr * f(F_IK, s) : 0.f;
                    ev[c + u] = x[u] * qk[u];
                    er += ev[c + u];
                }
                store16<T>(sb + S_DS, r, qc * 16 + c, x);
            }
            f(F_ER0 + qc, r) = er;
            const float cs = colsum16(ev, lane);
            if (lane < 16) f(F_EC0 + (warp & 1), qc * 16 + lane) = cs;
        } else {
            // dW = -(dDelta h^T) rows; dk += e^{Gl - G_r} Delta dH'^T
            const uint32_t wblk = (qc >> 1) ? S_DW1 : S_DW0;
            const float el = f(F_EL, r);
            float z = 0.f;  // e^{Gl-G_r} <(Delta dH'^T)_r, k_r>: dG terms of the decayed keys
#pragma unroll
            for (int c = 0; c < 32; c += 16) {
                float x[16], y[16], kv[16];
                umma::ld16(umma::taddr(tmem, lb, T_R1 + qc * 32 + c), x);
                umma::ld16(umma::taddr(tmem, lb, T_R2 + qc * 32 + c), y);
                load16<T>(sb + S_K0 + (qc >> 1) * 16384, r, (qc & 1) * 32 + c, kv);
                umma::ld_wait();
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    x[u] = -x[u];
                    acc[c + u] += el * y[u];
                    z += el * y[u] * kv[u];
                }
                store16<T>(sb + wblk, r, (qc & 1) * 32 + c, x);
            }
            f(F_Z0 + qc, r) = z * f(F_IK, r);
        }
        sync_tc();

        // ---------------- round 2
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) umma::mma(tmem + T_R1, dAmn + ks * 128, dDDmn + ks * 128, i_n256_mn, ks > 0);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t ko = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
                umma::mma(tmem + T_R8, dWup + ko, dKa + ko, i_n64, ks > 0);
            }
            umma::commit(bar);
        }
        // h, dH' and dO are free: the next unit's first tile group
        if (wn >= 0) {
            if (tid == TT) issue(nxt, jn, 1);
            posted = true;
            fetch_gates(nxt);
        }
        if (!wait_mma()) {
            ok = false;
            break;
        }
        if (!upper) {
            float vd = 0.f, kd = 0.f;
            // dDelta-side: ddelta = A^T dDelta (columns 0..127), A^T dW (128..255)
            const float br = f(F_B, r);
            T *dvrow = static_cast<T *>(p.dv) + ((tok0 + r) * Hv + j) * geo.V + qc * 32;
#pragma unroll
            for (int c = 0; c < 32; c += 16) {
                float x[16], y[16], vv[16], kv[16];
                umma::ld16(umma::taddr(tmem, lb, T_R1 + qc * 32 + c), x);
                umma::ld16(umma::taddr(tmem, lb, T_R1 + 128 + qc * 32 + c), y);
                load16<T>(sb + S_V0 + (qc >> 1) * 16384, r, (qc & 1) * 32 + c, vv);
                load16<T>(sb + S_K0 + (qc >> 1) * 16384, r, (qc & 1) * 32 + c, kv);
                umma::ld_wait();
                uint32_t w[8];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    vd += vv[u] * x[u];
                    kd += kv[u] * y[u];
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) w[u] = Elt<T>::pack(x[2 * u] * br, x[2 * u + 1] * br);
                if (valid == C) {
                    const uint32_t stg = sb + ((qc >> 1) ? S_DW1 : S_DW0);
                    const int col = (qc & 1) * 32 + c;  // (16-byte aligned)
                    umma::st_shared_v4(stg + umma::off(r, col, 0), w[0], w[1], w[2], w[3]);
                    umma::st_shared_v4(stg + umma::off(r, col + 8, 0), w[4], w[5], w[6], w[7]);
                } else if (r < valid) {
                    if (qc * 32 + c < geo.V) *reinterpret_cast<uint4 *>(dvrow + c) = make_uint4(w[0], w[1], w[2], w[3]);
                    if (qc * 32 + c + 8 < geo.V)
                        *reinterpret_cast<uint4 *>(dvrow + c + 8) = make_uint4(w[4], w[5], w[6], w[7]);
                }
            }
            f(F_VD0 + qc, r) = vd;
            f(F_KD0 + qc, r) = kd * f(F_IK, r);  // <k^_r, .>
            if (valid == C) {
                umma::fence_async_smem();
                asm volatile("bar.sync 2, 256;\n" ::: "memory");  // the eight lower-lane warps
                if (tid == ST) {
                    tma::store3d(&p.tdv, 0, j, (int)tok0, sb + S_DW0);
                    if (geo.V > 64) tma::store3d(&p.tdv, 64, j, (int)tok0, sb + S_DW1);
                    tma::commit_group();
                }
            }
        } else {
            // dk += diag(beta e^G) A^T dW ; dA = beta_s (e^{G_s} dW K^^T + dDelta V^T), strictly lower
            const float bg = f(F_B, r) * f(F_EG, r);
#pragma unroll
            for (int c = 0; c < 32; c += 16) {
                float x[16];
                umma::ld16(umma::taddr(tmem, lb, T_R1 + 128 + qc * 32 + c), x);
                umma::ld_wait();
#pragma unroll
                for (int u = 0; u < 16; ++u) acc[c + u] += bg * x[u];
            }
            {
                const int c = 0;
                float x1[16], x2[16];
                umma::ld16(umma::taddr(tmem, lb, T_R8 + qc * 16), x1);
                umma::ld16(umma::taddr(tmem, lb, T_R3 + qc * 16), x2);
                umma::ld_wait();
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int s = qc * 16 + u;
                    x1[u] = (s < r && r < valid) ? f(F_B, s) * (f(F_EG, s) * f(F_IK, s) * x1[u] + x2[u]) : 0.f;
                }
                store16<T>(sb + S_DA, r, qc * 16 + c, x1);
            }
        }
        sync_tc();

        // ---------------- round 3: X = dA A^T ; dq += dS K^ = diag(1/nq) dS'' K ; dk += dS^T Q^ = diag(1/nk) dS''^T Q
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                umma::mma(tmem + T_R8, dDA + ks * 2, dAk + ks * 2, i_n64, ks > 0);
                umma::mma(tmem + T_R1, dDS + ks * 2, dKmn + ks * 128, i_n128_bmn, ks > 0);
                umma::mma(tmem + T_R2, dDSup + ks * 128, dQmn + ks * 128, i_n128_mn, ks > 0);
            }
            umma::commit(bar);
            // V and dDelta are free (round 3 reads V's second block only as the unread partner rows of dA)
            if (wn >= 0) issue(nxt, jn, 2);
        }
        if (!wait_mma()) {
            ok = false;
            break;
        }
        if (!upper) {
            {
                float x[16];
                umma::ld16(umma::taddr(tmem, lb, T_R8 + qc * 16), x);
                umma::ld_wait();
                store16<T>(sb + S_X, r, qc * 16, x);
            }
            const float mq = f(F_MQ, r);
#pragma unroll
            for (int c = 0; c < 32; c += 16) {
                float x[16];
                umma::ld16(umma::taddr(tmem, lb, T_R1 + qc * 32 + c), x);
                umma::ld_wait();
#pragma unroll
                for (int u = 0; u < 16; ++u) acc[c + u] += mq * x[u];
            }
        } else {
            const float mk = f(F_MK, r);
#pragma unroll
            for (int c = 0; c < 32; c += 16) {
                float x[16];
                umma::ld16(umma::taddr(tmem, lb, T_R2 + qc * 32 + c), x);
                umma::ld_wait();
#pragma unroll
                for (int u = 0; u < 16; ++u) acc[c + u] += mk * x[u];
            }
        }
        sync_tc();

        // ---------------- round 4: dL = -A^T X
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) umma::mma(tmem + T_R8, dAup + ks * 128, dXmn + ks * 128, i_n64_mn, ks > 0);
            umma::commit(bar);
            if (wn >= 0) issue(nxt, jn, 3);  // round 3 has read dA: Delta's first block is free
        }
        if (!wait_mma()) {
            ok = false;
            break;
        }
        float lb_ = 0.f;  // upper lanes: sum_s dL Gamma K^K^^T
        if (upper) {
            // dKK = dL o beta_r Gamma, stored as dKK'' = diag(nk) dKK diag(nk) for the raw-tile products of
            // round 5; K^K^^T = nk_r nk_s (K K^T)
            const float gr = f(F_G, r), br = f(F_B, r), nkr = f(F_IK, r);
            float fv[16], fr = 0.f;  // F = dL o L: decay terms of dG
            {
                const int c = 0;
                float x[16], kk[16];
                umma::ld16(umma::taddr(tmem, lb, T_R8 + qc * 16), x);
                umma::ld16(umma::taddr(tmem, lb, T_R4 + qc * 16), kk);
                umma::ld_wait();
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int s = qc * 16 + u;
                    const bool m = s < r && r < valid;
                    const float gam = m ? __expf(gr - f(F_G, s)) : 0.f;
                    const float dlv = m ? -x[u] : 0.f;
                    const float nks = f(F_IK, s), kkh = kk[u] * nkr * nks;
                    lb_ += dlv * gam * kkh;
                    const float dkk = dlv * br * gam;
                    fv[c + u] = dkk * kkh;
                    fr += fv[c + u];
                    x[u] = dkk * nkr * nks;
                }
                store16<T>(sb + S_DKK, r, qc * 16 + c, x);
            }
            f(F_FR0 + qc, r) = fr;
            const float cs = colsum16(fv, lane);
            if (lane < 16) f(F_FC0 + ((warp & 3) - 2), qc * 16 + lane) = cs;
        } else {
            if (warp < 2) {
                // the dG / dbeta terms known by now (all but F and the dKK ones), for rows 32 warp..:
                // dG_r = E row - E column + <q_r, dq_inter_r> - z_r + beta_r e^{G_r} <(A^T dW)_r, k_r> (+ F row
                // - F column at the end); dbeta_r = e^{G_r} <(A^T dW)_r, k_r> + <(A^T dDelta)_r, v_r> (+ the
                // dKK term at the end); and this warp's share of sum_s z_s
                const int rr = warp * 32 + lane;
                auto q4 = [&](int slot0) {  // the four column-quarter partials, in a fixed order
                    return (f(slot0, rr) + f(slot0 + 1, rr)) + (f(slot0 + 2, rr) + f(slot0 + 3, rr));
                };
                const float z = q4(F_Z0), kd2 = q4(F_KD0);
                f(F_PDG, rr) = q4(F_ER0) - (f(F_EC0, rr) + f(F_EC0 + 1, rr)) + q4(F_QD0) - z +
                               f(F_B, rr) * f(F_EG, rr) * kd2;
                f(F_PDB, rr) = f(F_EG, rr) * kd2 + q4(F_VD0);
                float zs = rr < valid ? z : 0.f;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) zs += __shfl_xor_sync(0xffffffffu, zs, o);
                if (lane == 0) f(F_DG, 2 * warp) = zs;
                if (warp == 0 && lane == 0) {
                    float hd = 0.f;
#pragma unroll
                    for (int wi = 0; wi < 8; ++wi) hd += f(F_HD, wi);
                    f(F_DG, 4) = hd;
                }
            }
        }
        if (!upper && last_head) {
            // dq is complete after round 3: the lower-lane warps store it while the upper ones work on dKK
            if (p.l2norm) dot_partial();
            if (tid == ST) tma::wait_read();  // dv's staging block dW0 is free again
            asm volatile("bar.sync 2, 256;\n" ::: "memory");  // the eight lower-lane warps
            store_row(tok0, valid, hq);
            umma::fence_async_smem();
            asm volatile("bar.sync 2, 256;\n" ::: "memory");
            if (tid == ST) {
                if (valid == C) {
                    tma::store3d(&p.tdq, 0, hq, (int)tok0, sb + S_X);
                    if (geo.K > 64) tma::store3d(&p.tdq, 64, hq, (int)tok0, sb + S_DW0);
                    tma::commit_group();
                }
                if (wn >= 0) issue(nxt, jn, 5);  // the q tile has been read for the last time
            }
        }
        sync_tc();

        // ---------------- round 5: dk += dKK K^ + dKK^T K^ = diag(1/nk) (dKK'' K + dKK''^T K)
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                umma::mma(tmem + T_R1, dKKk + ks * 2, dKmn + ks * 128, i_n128_bmn, ks > 0);
                umma::mma(tmem + T_R1, dKKmn + ks * 128, dKmn + ks * 128, i_n128_mn, true);
            }
            umma::commit(bar);
            if (wn >= 0) issue(nxt, jn, 4);  // round 4 has read A
        }
        if (!wait_mma()) {
            ok = false;
            break;
        }
        if (upper) {
            const float mk = f(F_MK, r);
#pragma unroll
            for (int c = 0; c < 32; c += 16) {
                float x[16];
                umma::ld16(umma::taddr(tmem, lb, T_R1 + qc * 32 + c), x);
                umma::ld_wait();
#pragma unroll
                for (int u = 0; u < 16; ++u) acc[c + u] += mk * x[u];
            }
            f(F_LB0 + qc, r) = lb_;
        }
        // dk's partial dot products of the L2-norm chain rule go with the round-5 results, so one barrier
        // serves both the dG reduction and the dk stores
        if (upper && last_head && p.l2norm) dot_partial();
        __syncthreads();
        if (warp < 2) {
            // dG_r = (the round-4 partial) + F row - F column; every valid row's dg also carries
            // e^{Gl} <dH', h> + sum_s z_s (the last valid row's extra terms, summed backwards).  Warp w takes
            // rows 32w..32w+31.
            const int rr = warp * 32 + lane;
            const bool vr = rr < valid;
            auto q4 = [&](int slot0) {  // the four column-quarter partials, in a fixed order
                return (f(slot0, rr) + f(slot0 + 1, rr)) + (f(slot0 + 2, rr) + f(slot0 + 3, rr));
            };
            const float dG = f(F_PDG, rr) + q4(F_FR0) - (f(F_FC0, rr) + f(F_FC0 + 1, rr));
            if (vr) store_gate<T>(p.dbeta, (tok0 + rr) * Hv + j, p.gate_f32, f(F_PDB, rr) + q4(F_LB0));
            // dg_s = sum_{r >= s} dG_r within the chunk: suffix sums inside the warp, then warp 1's total
            float y = vr ? dG : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float t = __shfl_down_sync(0xffffffffu, y, o);
                if (lane + o < 32) y += t;
            }
            if (lane == 0) f(F_DG, 2 * warp + 1) = y;
            asm volatile("bar.sync 1, 64;\n" ::: "memory");  // warps 0 and 1
            const float extra = __expf(Gl) * f(F_DG, 4) + (f(F_DG, 0) + f(F_DG, 2));
            const float tail = warp == 0 ? f(F_DG, 3) : 0.f;
            if (vr) store_gate<T>(p.dg, (tok0 + rr) * Hv + j, p.gate_f32, y + tail + extra);
        }
        if (upper) {
            if (last_head) store_row(tok0, valid, hq);
            // k and Delta's second block are free once the upper-lane warps are done (the lower ones no longer
            // read them): the next unit's last tile group goes in while warps 0 and 1 finish dG
            umma::fence_async_smem();
            asm volatile("bar.sync 3, 256;\n" ::: "memory");  // the eight upper-lane warps
            if (tid == TT && wn >= 0) issue(nxt, jn, 6);
        }
        umma::fence_async_smem();
        __syncthreads();
        if (tid == ST && last_head && valid == C) {
            tma::store3d(&p.tdk, 0, hq, (int)tok0, sb + S_DS);
            if (geo.K > 64) tma::store3d(&p.tdk, 64, hq, (int)tok0, sb + S_DW1);
            tma::commit_group();
        }
        if (wn < 0) break;
        wit = wn;
        jj = jn;
        cur = nxt;
    }
    // after an error, let a prefetch in flight land before the block exits (bounded)
    if (tid == 0 && posted) umma::mbar_wait(lbar, lphase, 4000000L);
    if (tid == ST) tma::wait_all();  // the staged output rows are written before shared memory goes away

    umma::fence_before();
    __syncthreads();
    if (warp == 0) umma::dealloc(tmem, T_COLS);
}

template <typename T>
cudaError_t bwd_chunk_tc_t(const Args &a, const BcP &p, cudaStream_t s) {
    if (a.max_chunks == 0) return cudaSuccess;
    if ((long long)a.max_chunks * a.Hq >= (1ll << 31)) return cudaErrorInvalidValue;  // 32-bit item indices
    auto kern = bwd_chunk_tc_kernel<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S_BYTES);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const long items = (long)a.max_chunks * a.Hq;
    const unsigned grid = (unsigned)(items < sms ? items : sms);  // one persistent CTA per SM
    return launch_overlapped(kern, dim3(grid), dim3(NT), S_BYTES, s, make_geo(a), p);
}

}  // namespace

cudaError_t launch_bwd_chunk_tc(const Args &a, const void *q, const void *k, const void *v, const float *g_cs,
                                const void *beta, const void *A, const void *dout, const void *h, const void *dhn,
                                const void *delta, const void *ddelta, void *dq, void *dk, void *dv, void *dg,
                                void *dbeta, cudaStream_t s) {
    BcP p;
    const uint64_t tokens = (uint64_t)a.B * (uint64_t)a.T, rows = (uint64_t)a.max_chunks * a.Hv;
    const bool bf = a.bf16;
    if (!make_token_map(&p.tq, q, bf, a.K, a.Hq, tokens, 64) || !make_token_map(&p.tk, k, bf, a.K, a.Hq, tokens, 64) ||
        !make_token_map(&p.tdo, dout, bf, a.V, a.Hv, tokens, 64) || !make_token_map(&p.tv, v, bf, a.V, a.Hv, tokens, 64) ||
        !make_tmap_3d(&p.ta, A, bf, C, a.Hv, tokens, C * 2, (uint64_t)a.Hv * C * 2, 64, 1, 64) ||
        !make_tmap_3d(&p.th, h, bf, DV, DK, rows, DV * 2, (uint64_t)DK * DV * 2, 64, 128, 1) ||
        !make_tmap_3d(&p.tdh, dhn, bf, DV, DK, rows, DV * 2, (uint64_t)DK * DV * 2, 64, 128, 1) ||
        !make_tmap_3d(&p.td, delta, bf, DV, C, rows, DV * 2, (uint64_t)C * DV * 2, 64, 64, 1) ||
        !make_tmap_3d(&p.tdd, ddelta, bf, DV, C, rows, DV * 2, (uint64_t)C * DV * 2, 64, 64, 1) ||
        !make_token_map(&p.tdq, dq, bf, a.K, a.Hq, tokens, 64) || !make_token_map(&p.tdk, dk, bf, a.K, a.Hq, tokens, 64) ||
        !make_token_map(&p.tdv, dv, bf, a.V, a.Hv, tokens, 64))
        return cudaErrorInvalidValue;
    p.q = q;
    p.k = k;
    p.v = v;
    p.A = A;
    p.beta = beta;
    p.dout = dout;
    p.h = h;
    p.dhn = dhn;
    p.delta = delta;
    p.ddelta = ddelta;
    p.g_cs = g_cs;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.dbeta = dbeta;
    p.dg = dg;
    p.gate_f32 = a.gate_f32;
    p.l2norm = a.l2norm;
    p.scale = a.scale;
    p.nslots = (int)a.max_chunks;
    return a.bf16 ? bwd_chunk_tc_t<__nv_bfloat16>(a, p, s) : bwd_chunk_tc_t<__half>(a, p, s);
}

}  // namespace gdr
