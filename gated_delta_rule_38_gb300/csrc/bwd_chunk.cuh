// bwd_chunk: per-chunk gradients (included by bwd.cu inside namespace gdr).
//
// 8 warps: warp w owns token rows 16*(w&3).. and the column half (w>>2) of
// every product it computes.  Phases are separated by block barriers; each
// phase writes the operands of the next one to shared memory.

struct ChunkBwdP {
    const void *q, *k, *v, *A, *beta, *dout, *h, *dhn;
    const float *g_cs;
    void *dq, *dk, *dv, *dg, *dbeta;
    bool gate_f32, l2norm;
    float scale;
};

constexpr int BC_Q = 0, BC_K = 16384, BC_V = 32768, BC_DO = 49152, BC_A = 65536, BC_H = 73728, BC_DH = 106496,
              BC_D = 139264, BC_DD = 155648, BC_DS = 172032, BC_DW = 180224, BC_F = 196608;
constexpr int BC_DA = BC_H, BC_X = BC_H + 8192, BC_DKK = BC_H + 16384;  // reuse the state tile after phase 3
constexpr int NRED = 22;
constexpr int BC_SMEM = BC_F + (2 + NRED) * C * 4 + 8 * 4 + C * 4;

// red[] slots: row/column partial sums, reduced in a fixed order at the end.
enum {
    R_EROW = 0, R_ECOL = 2, R_QDOT = 6, R_Z = 8, R_KDOT = 10, R_VDOT = 12, R_DBL = 14, R_FROW = 16, R_FCOL = 18
};

// Sum of a 16 x (8*NT) fragment strip over its columns, per row -> out[R0 + row].
template <int NT>
__device__ __forceinline__ void row_partial(const float (*v)[4], float *out, int R0, int lane) {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        s0 += v[nt][0] + v[nt][1];
        s1 += v[nt][2] + v[nt][3];
    }
    s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
    if ((lane & 3) == 0) {
        out[R0 + (lane >> 2)] = s0;
        out[R0 + (lane >> 2) + 8] = s1;
    }
}

// Sum over the strip's 16 rows, per column -> out[C0 + col].
template <int NT>
__device__ __forceinline__ void col_partial(const float (*v)[4], float *out, int C0, int lane) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float s = v[nt][e] + v[nt][2 + e];
            s += __shfl_xor_sync(0xffffffffu, s, 4);
            s += __shfl_xor_sync(0xffffffffu, s, 8);
            s += __shfl_xor_sync(0xffffffffu, s, 16);
            if (lane < 4) out[C0 + nt * 8 + lane * 2 + e] = s;
        }
}

// Per-row dot product of a fragment strip with the same positions of a tile.
template <typename T, int NT>
__device__ __forceinline__ void row_dot(const float (*v)[4], const Tile &t, float *out, int R0, int C0, int lane) {
    const int gq = lane >> 2, tq = lane & 3;
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int col = C0 + nt * 8 + tq * 2;
        const float2 a = Elt<T>::unpack(lds32(t.addr(R0 + gq, col)));
        const float2 b = Elt<T>::unpack(lds32(t.addr(R0 + gq + 8, col)));
        s0 += v[nt][0] * a.x + v[nt][1] * a.y;
        s1 += v[nt][2] * b.x + v[nt][3] * b.y;
    }
    s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
    if (tq == 0) {
        out[R0 + gq] = s0;
        out[R0 + gq + 8] = s1;
    }
}

template <int NT>
__device__ __forceinline__ void scale_rows(float (*v)[4], float f0, float f1) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        v[nt][0] *= f0;
        v[nt][1] *= f0;
        v[nt][2] *= f1;
        v[nt][3] *= f1;
    }
}

// dx = (dxh - xh (xh . dxh)) / n with n = sqrt(sum x^2 + eps), xh = x / n, one warp per row;
// the fp32 gradient rows come from `src` ([64][128] fp32 in shared memory).
template <typename T>
__device__ __forceinline__ void l2norm_bwd_rows(const float *src, const T *x, long long stride, T *dst, int valid,
                                                bool l2norm, int warp, int nwarps, int lane) {
    for (int r = warp; r < valid; r += nwarps) {
        const T *xr = x + (long long)r * stride;
        T *dr = dst + (long long)r * stride;
        float xv[4], gv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            xv[u] = Elt<T>::to_f(xr[lane * 4 + u]);
            gv[u] = src[r * DK + lane * 4 + u];
        }
        if (l2norm) {
            float ss = xv[0] * xv[0] + xv[1] * xv[1] + xv[2] * xv[2] + xv[3] * xv[3];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            const float inv = 1.0f / sqrtf(ss + L2_EPS);
            float dot = 0.f;
#pragma unroll
            for (int u = 0; u < 4; ++u) dot += xv[u] * inv * gv[u];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
#pragma unroll
            for (int u = 0; u < 4; ++u) gv[u] = (gv[u] - xv[u] * inv * dot) * inv;
        }
        uint2 w;
        w.x = Elt<T>::pack(gv[0], gv[1]);
        w.y = Elt<T>::pack(gv[2], gv[3]);
        *reinterpret_cast<uint2 *>(dr + lane * 4) = w;
    }
}

template <typename T>
__global__ void __launch_bounds__(256, 1) bwd_chunk_kernel(Geo geo, ChunkBwdP p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    long long tok0;
    int valid, n, ci;
    const int slot = blockIdx.x;
    if (!geo.chunk(slot, tok0, valid, n, ci)) return;
    const int hq = blockIdx.y, Hv = geo.Hv, Hq = geo.Hq, grp = Hv / Hq;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, tq = lane & 3;
    const int rs = warp & 3, ch = warp >> 2, R0 = rs * 16;
    const T *q = static_cast<const T *>(p.q);
    const T *k = static_cast<const T *>(p.k);
    const T *v = static_cast<const T *>(p.v);
    const T *A = static_cast<const T *>(p.A);
    const T *dout = static_cast<const T *>(p.dout);
    const T *hs = static_cast<const T *>(p.h);
    const T *dhs = static_cast<const T *>(p.dhn);

    const Tile sQ = make_tile(smem + BC_Q, DK), sK = make_tile(smem + BC_K, DK), sV = make_tile(smem + BC_V, DV);
    const Tile sdO = make_tile(smem + BC_DO, DV), sA = make_tile(smem + BC_A, C), sH = make_tile(smem + BC_H, DV);
    const Tile sDH = make_tile(smem + BC_DH, DV), sD = make_tile(smem + BC_D, DV), sdD = make_tile(smem + BC_DD, DV);
    const Tile sdS = make_tile(smem + BC_DS, C), sdW = make_tile(smem + BC_DW, DK);
    const Tile sdA = make_tile(smem + BC_DA, C), sX = make_tile(smem + BC_X, C), sdKK = make_tile(smem + BC_DKK, C);
    float *sG = reinterpret_cast<float *>(smem + BC_F);
    float *sB = sG + C;
    float *red = sB + C;           // [NRED][64]
    float *hred = red + NRED * C;  // [8]

    load_rows_async<T>(sQ, q + (tok0 * Hq + hq) * DK, (long long)Hq * DK, C, valid, DK, tid, 256);
    load_rows_async<T>(sK, k + (tok0 * Hq + hq) * DK, (long long)Hq * DK, C, valid, DK, tid, 256);
    cp_async_commit();

    float dqa[8][4], dka[8][4];
    zero_acc<8>(dqa);
    zero_acc<8>(dka);
    bool first = true;

    for (int jj = 0; jj < grp; ++jj) {
        const int j = hq * grp + jj;
        const long long sbase = ((long long)slot * Hv + j) * DK * DV;
        load_rows_async<T>(sV, v + (tok0 * Hv + j) * DV, (long long)Hv * DV, C, valid, DV, tid, 256);
        load_rows_async<T>(sdO, dout + (tok0 * Hv + j) * DV, (long long)Hv * DV, C, valid, DV, tid, 256);
        load_rows_async<T>(sA, A + (tok0 * Hv + j) * C, (long long)Hv * C, C, valid, C, tid, 256);
        load_rows_async<T>(sH, hs + sbase, DV, DK, DK, DV, tid, 256);
        load_rows_async<T>(sDH, dhs + sbase, DV, DK, DK, DV, tid, 256);
        if (tid < C) {
            const bool ok = tid < valid;
            cp_async4b(smem_u32(sG + tid), p.g_cs + (ok ? (tok0 + tid) * Hv + j : 0), ok);
            sB[tid] = ok ? load_gate<T>(p.beta, (tok0 + tid) * Hv + j, p.gate_f32) : 0.f;
        }
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
        if (first) {
            if (p.l2norm) {
                l2norm_rows<T>(sQ, valid, warp, 8, lane);
                l2norm_rows<T>(sK, valid, warp, 8, lane);
                __syncthreads();
            }
            first = false;
        }
        const float Gl = sG[valid - 1];
        const float Gr0 = sG[R0 + gq], Gr1 = sG[R0 + gq + 8];

        // ---- P1: Delta = A diag(beta) V - A diag(beta e^G) K h   (rows R0, value half ch)
        {
            uint32_t ab[4][4], akg[4][4];
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                uint32_t a[4];
                load_a(a, sA, R0, ks * 16, false, lane);
                scale_cols2<T>(ab[ks], a, sB, sG, false, ks * 16, tq);
                scale_cols2<T>(akg[ks], a, sB, sG, true, ks * 16, tq);
            }
            uint32_t wf[8][4];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float wacc[8][4];
                zero_acc<8>(wacc);
                warp_mma_ra<T, 8, 4>(wacc, akg, sK, half * 64, true, 0, lane);
                acc_to_a<T, 4>(&wf[half * 4], wacc, -1.f);
            }
            float dacc[8][4];
            zero_acc<8>(dacc);
            warp_mma_ra<T, 8, 4>(dacc, ab, sV, ch * 64, true, 0, lane);
            warp_mma_ra<T, 8, 8>(dacc, wf, sH, ch * 64, true, 0, lane);
            store_acc<T, 8>(sD, dacc, R0, ch * 64, lane);
        }
        __syncthreads();

        // ---- P2a: dDelta = e^{Gl-G_r} (K dH')_r + scale (P^T dO)_r   (rows R0, value half ch)
        {
            float acc[8][4];
            zero_acc<8>(acc);
            warp_mma<T, 8, 8>(acc, sK, R0, false, sDH, ch * 64, true, 0, lane);
            scale_rows<8>(acc, __expf(Gl - Gr0), __expf(Gl - Gr1));
            float pacc[8][4];
            zero_acc<8>(pacc);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                uint32_t a[4];
                load_a(a, sK, R0, ks * 16, false, lane);
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    if (np >= rs) {
                        uint32_t b[4];
                        load_b2(b, sQ, np * 16, ks * 16, false, lane);
                        mma16816<T>(pacc[2 * np], a, b[0], b[1]);
                        mma16816<T>(pacc[2 * np + 1], a, b[2], b[3]);
                    }
                }
            }
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = R0 + gq + (e >> 1) * 8, s = nt * 8 + tq * 2 + (e & 1);
                    pacc[nt][e] = (s >= r && s < valid) ? pacc[nt][e] * p.scale * __expf(sG[s] - sG[r]) : 0.f;
                }
            uint32_t pt[4][4];
            acc_to_a<T, 4>(pt, pacc);
            warp_mma_ra<T, 8, 4>(acc, pt, sdO, ch * 64, true, 0, lane);
            store_acc<T, 8>(sdD, acc, R0, ch * 64, lane);
        }
        // ---- P2b: dP = scale dO Delta^T, P = Q K^T o Gamma (rows R0, key-token half ch)
        {
            float dp[4][4], pp[4][4];
            zero_acc<4>(dp);
            zero_acc<4>(pp);
            warp_mma<T, 4, 8>(dp, sdO, R0, false, sD, ch * 32, false, 0, lane);
            warp_mma<T, 4, 8>(pp, sQ, R0, false, sK, ch * 32, false, 0, lane);
            float E[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int r = R0 + gq + hh * 8;
                    float ds[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int s = ch * 32 + nt * 8 + tq * 2 + e;
                        const bool m = s <= r && r < valid;
                        const float gam = m ? __expf(sG[r] - sG[s]) : 0.f;
                        const float dpv = p.scale * dp[nt][2 * hh + e];
                        ds[e] = dpv * gam;
                        E[nt][2 * hh + e] = ds[e] * pp[nt][2 * hh + e];
                    }
                    sts32(sdS.addr(r, ch * 32 + nt * 8 + tq * 2), Elt<T>::pack(ds[0], ds[1]));
                }
            }
            row_partial<4>(E, red + (R_EROW + ch) * C, R0, lane);
            col_partial<4>(E, red + (R_ECOL + rs) * C, ch * 32, lane);
        }
        __syncthreads();

        // ---- P3: dQ, dK from P and the state; dW
        {
            float acc[8][4];
            zero_acc<8>(acc);
            warp_mma<T, 8, 8>(acc, sdO, R0, false, sH, ch * 64, false, 0, lane);
            scale_rows<8>(acc, p.scale * __expf(Gr0), p.scale * __expf(Gr1));
            row_dot<T, 8>(acc, sQ, red + (R_QDOT + ch) * C, R0, ch * 64, lane);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) dqa[nt][e] += acc[nt][e];
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                if (ks <= rs) warp_mma<T, 8, 1>(dqa, sdS, R0, false, sK, ch * 64, true, ks * 16, lane);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                if (ks >= rs) warp_mma<T, 8, 1>(dka, sdS, R0, true, sQ, ch * 64, true, ks * 16, lane);
            zero_acc<8>(acc);
            warp_mma<T, 8, 8>(acc, sD, R0, false, sDH, ch * 64, false, 0, lane);
            scale_rows<8>(acc, __expf(Gl - Gr0), __expf(Gl - Gr1));
            row_dot<T, 8>(acc, sK, red + (R_Z + ch) * C, R0, ch * 64, lane);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) dka[nt][e] += acc[nt][e];
            zero_acc<8>(acc);
            warp_mma<T, 8, 8>(acc, sdD, R0, false, sH, ch * 64, false, 0, lane);
            store_acc<T, 8>(sdW, acc, R0, ch * 64, lane, -1.f);
            // <dH', h> over the whole state: both tiles share one swizzle, so equal offsets hold equal elements
            float hd = 0.f;
            const uint32_t hb = smem_u32(smem + BC_H), db = smem_u32(smem + BC_DH);
#pragma unroll 4
            for (int u = 0; u < 32; ++u) {
                const uint32_t off = (uint32_t)(tid * 32 + u) * 4u;
                const float2 a = Elt<T>::unpack(lds32(hb + off));
                const float2 b = Elt<T>::unpack(lds32(db + off));
                hd += a.x * b.x + a.y * b.y;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) hd += __shfl_xor_sync(0xffffffffu, hd, o);
            if (lane == 0) hred[warp] = hd;
        }
        __syncthreads();

        // ---- P4: dA, A^T dW, A^T dDelta (dV)
        {
            float a1[4][4], a2[4][4];
            zero_acc<4>(a1);
            zero_acc<4>(a2);
            warp_mma<T, 4, 8>(a1, sdW, R0, false, sK, ch * 32, false, 0, lane);
            warp_mma<T, 4, 8>(a2, sdD, R0, false, sV, ch * 32, false, 0, lane);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int r = R0 + gq + hh * 8;
                    float w2[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int s = ch * 32 + nt * 8 + tq * 2 + e;
                        const bool m = s < r && r < valid;
                        w2[e] = m ? sB[s] * (a1[nt][2 * hh + e] * __expf(sG[s]) + a2[nt][2 * hh + e]) : 0.f;
                    }
                    sts32(sdA.addr(r, ch * 32 + nt * 8 + tq * 2), Elt<T>::pack(w2[0], w2[1]));
                }
            float acc[8][4];
            zero_acc<8>(acc);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                if (ks >= rs) warp_mma<T, 8, 1>(acc, sA, R0, true, sdW, ch * 64, true, ks * 16, lane);
            row_dot<T, 8>(acc, sK, red + (R_KDOT + ch) * C, R0, ch * 64, lane);
            const float b0 = sB[R0 + gq] * __expf(Gr0), b1 = sB[R0 + gq + 8] * __expf(Gr1);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                dka[nt][0] += acc[nt][0] * b0;
                dka[nt][1] += acc[nt][1] * b0;
                dka[nt][2] += acc[nt][2] * b1;
                dka[nt][3] += acc[nt][3] * b1;
            }
            zero_acc<8>(acc);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                if (ks >= rs) warp_mma<T, 8, 1>(acc, sA, R0, true, sdD, ch * 64, true, ks * 16, lane);
            row_dot<T, 8>(acc, sV, red + (R_VDOT + ch) * C, R0, ch * 64, lane);
            T *dv = static_cast<T *>(p.dv);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = R0 + gq + hh * 8;
                if (r < valid) {
                    const float br = sB[r];
                    T *row = dv + ((tok0 + r) * Hv + j) * DV + ch * 64;
#pragma unroll
                    for (int nt = 0; nt < 8; ++nt)
                        *reinterpret_cast<uint32_t *>(row + nt * 8 + tq * 2) =
                            Elt<T>::pack(acc[nt][2 * hh] * br, acc[nt][2 * hh + 1] * br);
                }
            }
        }
        __syncthreads();

        // ---- P5: X = dA A^T
        {
            float acc[4][4];
            zero_acc<4>(acc);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                if (ks <= rs) warp_mma<T, 4, 1>(acc, sdA, R0, false, sA, ch * 32, false, ks * 16, lane);
            store_acc<T, 4>(sX, acc, R0, ch * 32, lane);
        }
        __syncthreads();

        // ---- P6: dL = -A^T X (strictly lower), dKK = dL o beta_r Gamma, dbeta and dG terms of L
        {
            float acc[4][4], kk[4][4];
            zero_acc<4>(acc);
            zero_acc<4>(kk);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                if (ks >= rs) warp_mma<T, 4, 1>(acc, sA, R0, true, sX, ch * 32, true, ks * 16, lane);
            warp_mma<T, 4, 8>(kk, sK, R0, false, sK, ch * 32, false, 0, lane);
            float F[4][4], Db[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int r = R0 + gq + hh * 8;
                    float w2[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int s = ch * 32 + nt * 8 + tq * 2 + e;
                        const bool m = s < r && r < valid;
                        const float gam = m ? __expf(sG[r] - sG[s]) : 0.f;
                        const float dl = m ? -acc[nt][2 * hh + e] : 0.f;
                        const float kv = kk[nt][2 * hh + e];
                        w2[e] = dl * sB[r] * gam;
                        Db[nt][2 * hh + e] = dl * gam * kv;
                        F[nt][2 * hh + e] = dl * sB[r] * gam * kv;
                    }
                    sts32(sdKK.addr(r, ch * 32 + nt * 8 + tq * 2), Elt<T>::pack(w2[0], w2[1]));
                }
            row_partial<4>(Db, red + (R_DBL + ch) * C, R0, lane);
            row_partial<4>(F, red + (R_FROW + ch) * C, R0, lane);
            col_partial<4>(F, red + (R_FCOL + rs) * C, ch * 32, lane);
        }
        __syncthreads();

        // ---- P7: dK += dKK K + dKK^T K; then dG -> dg (reverse cumsum) and dbeta
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            if (ks <= rs) warp_mma<T, 8, 1>(dka, sdKK, R0, false, sK, ch * 64, true, ks * 16, lane);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            if (ks >= rs) warp_mma<T, 8, 1>(dka, sdKK, R0, true, sK, ch * 64, true, ks * 16, lane);
        if (warp == 0) {
            float zs = 0.f, dgv[2], dbv[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = lane + 32 * hh;
                const float z = red[(R_Z + 0) * C + r] + red[(R_Z + 1) * C + r];
                zs += z;
                const float eg = __expf(sG[r]);
                const float kd = red[(R_KDOT + 0) * C + r] + red[(R_KDOT + 1) * C + r];
                float dG = (red[(R_EROW + 0) * C + r] + red[(R_EROW + 1) * C + r]) -
                           (red[(R_ECOL + 0) * C + r] + red[(R_ECOL + 1) * C + r] + red[(R_ECOL + 2) * C + r] +
                            red[(R_ECOL + 3) * C + r]) +
                           (red[(R_QDOT + 0) * C + r] + red[(R_QDOT + 1) * C + r]) - z + sB[r] * eg * kd +
                           (red[(R_FROW + 0) * C + r] + red[(R_FROW + 1) * C + r]) -
                           (red[(R_FCOL + 0) * C + r] + red[(R_FCOL + 1) * C + r] + red[(R_FCOL + 2) * C + r] +
                            red[(R_FCOL + 3) * C + r]);
                dgv[hh] = r < valid ? dG : 0.f;
                dbv[hh] = eg * kd + (red[(R_VDOT + 0) * C + r] + red[(R_VDOT + 1) * C + r]) +
                          (red[(R_DBL + 0) * C + r] + red[(R_DBL + 1) * C + r]);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) zs += __shfl_xor_sync(0xffffffffu, zs, o);
            float hd = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) hd += hred[w];
            const float extra = __expf(Gl) * hd + zs;  // terms of G at the last valid row
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
                if (lane + 32 * hh == valid - 1) dgv[hh] += extra;
            // dg_s = sum_{r >= s} dG_r  (suffix sums over 64 rows held as two halves)
            float y1 = dgv[1], y0 = dgv[0];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float t1 = __shfl_down_sync(0xffffffffu, y1, o);
                const float t0 = __shfl_down_sync(0xffffffffu, y0, o);
                if (lane + o < 32) {
                    y1 += t1;
                    y0 += t0;
                }
            }
            y0 += __shfl_sync(0xffffffffu, y1, 0);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = lane + 32 * hh;
                if (r < valid) {
                    store_gate<T>(p.dg, (tok0 + r) * Hv + j, p.gate_f32, hh ? y1 : y0);
                    store_gate<T>(p.dbeta, (tok0 + r) * Hv + j, p.gate_f32, dbv[hh]);
                }
            }
        }
        __syncthreads();
    }

    // ---- dq, dk: stage the fp32 sums, apply the L2-norm chain rule, store
    float *fq = reinterpret_cast<float *>(smem + BC_V);  // [64][128] fp32 (V and dO tiles are free now)
    float *fk = reinterpret_cast<float *>(smem + BC_H);  // [64][128] fp32 (state tiles are free now)
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int r = R0 + gq + (e >> 1) * 8, c = ch * 64 + nt * 8 + tq * 2 + (e & 1);
            fq[r * DK + c] = dqa[nt][e];
            fk[r * DK + c] = dka[nt][e];
        }
    __syncthreads();
    const long long rstride = (long long)Hq * DK;
    l2norm_bwd_rows<T>(fq, q + (tok0 * Hq + hq) * DK, rstride, static_cast<T *>(p.dq) + (tok0 * Hq + hq) * DK, valid,
                       p.l2norm, warp, 8, lane);
    l2norm_bwd_rows<T>(fk, k + (tok0 * Hq + hq) * DK, rstride, static_cast<T *>(p.dk) + (tok0 * Hq + hq) * DK, valid,
                       p.l2norm, warp, 8, lane);
}

template <typename T>
static cudaError_t bwd_chunk_t(const Args &a, const ChunkBwdP &p, cudaStream_t s) {
    if (a.max_chunks == 0) return cudaSuccess;
    auto kern = bwd_chunk_kernel<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, BC_SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)a.max_chunks, a.Hq);
    kern<<<grid, 256, BC_SMEM, s>>>(make_geo(a), p);
    return cudaGetLastError();
}

cudaError_t launch_bwd_chunk(const Args &a, const void *q, const void *k, const void *v, const float *g_cs,
                             const void *beta, const void *A, const void *dout, const void *h, const void *dhn,
                             void *dq, void *dk, void *dv, void *dg, void *dbeta, cudaStream_t s) {
    ChunkBwdP p;
    p.q = q;
    p.k = k;
    p.v = v;
    p.A = A;
    p.beta = beta;
    p.dout = dout;
    p.h = h;
    p.dhn = dhn;
    p.g_cs = g_cs;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.dg = dg;
    p.dbeta = dbeta;
    p.gate_f32 = a.gate_f32;
    p.l2norm = a.l2norm;
    p.scale = a.scale;
    return a.bf16 ? bwd_chunk_t<__nv_bfloat16>(a, p, s) : bwd_chunk_t<__half>(a, p, s);
}
