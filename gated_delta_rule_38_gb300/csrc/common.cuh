// Shared device helpers for the gated delta rule kernels (sm_103a).
//
// Tiles of 16-bit elements live in shared memory row-major with rows of a
// multiple of 64 elements (128 bytes); the 16-byte chunk index inside a row
// is XOR-swizzled with (row & 7), so that 8 consecutive rows of the same
// logical chunk fall in 8 different bank groups (conflict-free ldmatrix and
// fragment stores).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "gdr.h"
#include "launch.h"

namespace gdr {

constexpr int C = GDR_CHUNK;  // tokens per chunk
constexpr int DK = 128;       // key head dim
constexpr int DV = 128;       // value head dim
constexpr float L2_EPS = 1e-6f;

// ---------------------------------------------------------------- element types

template <typename T> struct Elt;
template <> struct Elt<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
    static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&v);
    }
    static __device__ __forceinline__ float2 unpack(uint32_t u) {
        __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&u);
        return __bfloat1622float2(v);
    }
};
template <> struct Elt<__half> {
    static __device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
    static __device__ __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&v);
    }
    static __device__ __forceinline__ float2 unpack(uint32_t u) {
        __half2 v = *reinterpret_cast<__half2 *>(&u);
        return __half22float2(v);
    }
};

// Programmatic dependent launch (kernels launched by launch_overlapped): the next kernel in the stream may
// start launching once every block of this one has called griddep_launch_next; griddep_wait returns once
// the previous kernel has completed and its memory is visible, so it precedes every global memory access.
// Outside such a launch both are no-ops.
__device__ __forceinline__ void griddep_launch_next() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

// Gate-like per-token scalar (g, beta): the element type or fp32.
template <typename T>
__device__ __forceinline__ float load_gate(const void *p, long long i, bool f32) {
    return f32 ? static_cast<const float *>(p)[i] : Elt<T>::to_f(static_cast<const T *>(p)[i]);
}
template <typename T>
__device__ __forceinline__ void store_gate(void *p, long long i, bool f32, float x) {
    if (f32)
        static_cast<float *>(p)[i] = x;
    else
        static_cast<T *>(p)[i] = Elt<T>::from_f(x);
}

// ---------------------------------------------------------------- tensor-core fragments
// mma.sync m16n8k16, fp32 accumulate.  Fragment ownership (g = lane/4, t = lane%4):
//   A (16x16): a0 (g, 2t..2t+1) a1 (g+8, 2t..) a2 (g, 2t+8..) a3 (g+8, 2t+8..)
//   B (16x8) : b0 (k=2t..2t+1, n=g) b1 (k=2t+8.., n=g)
//   C (16x8) : c0,c1 (g, 2t..2t+1)  c2,c3 (g+8, 2t..2t+1)

template <typename T> __device__ __forceinline__ void mma16816(float *c, const uint32_t *a, uint32_t b0, uint32_t b1);
template <>
__device__ __forceinline__ void mma16816<__nv_bfloat16>(float *c, const uint32_t *a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<__half>(float *c, const uint32_t *a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// tf32 m16n8k8 (used for the triangular-inverse merges, fp32 operands).
//   A (16x8): a0 (g, t) a1 (g+8, t) a2 (g, t+4) a3 (g+8, t+4);  B (8x8): b0 (k=t, n=g) b1 (k=t+4, n=g)
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void mma1688_tf32(float *c, const uint32_t *a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t *r, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t *r, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- swizzled tiles

// A [rows x cols] tile of 16-bit values; cols is a multiple of 64.
struct Tile {
    uint32_t base;  // shared-space byte address
    int chunks;     // 16-byte chunks per row (= cols / 8)
    __device__ __forceinline__ uint32_t addr(int row, int col) const {
        const int ch = (col >> 3) ^ (row & 7);
        return base + (uint32_t)(row * chunks + ch) * 16u + (uint32_t)(col & 7) * 2u;
    }
};

__device__ __forceinline__ Tile make_tile(void *smem, int cols) { return Tile{smem_u32(smem), cols / 8}; }

// A fragment (16x16 at rows m0, cols k0) of the operand A[m][k].
//   trans = false: the tile stores A as [m][k];  trans = true: the tile stores [k][m].
__device__ __forceinline__ void load_a(uint32_t *a, const Tile &t, int m0, int k0, bool trans, int lane) {
    const int mat = lane >> 3, r8 = lane & 7;
    if (!trans) {
        ldsm_x4(a, t.addr(m0 + r8 + (mat & 1) * 8, k0 + (mat >> 1) * 8));
    } else {
        ldsm_x4_t(a, t.addr(k0 + r8 + (mat >> 1) * 8, m0 + (mat & 1) * 8));
    }
}

// B fragments of two adjacent n-tiles (n0..n0+15) at k0 of the operand B[k][n]:
//   b[0],b[1] for n-tile n0, b[2],b[3] for n-tile n0+8.
//   trans = false: the tile stores [n][k] (K contiguous);  trans = true: the tile stores [k][n].
__device__ __forceinline__ void load_b2(uint32_t *b, const Tile &t, int n0, int k0, bool trans, int lane) {
    const int mat = lane >> 3, r8 = lane & 7;
    if (!trans) {
        ldsm_x4(b, t.addr(n0 + r8 + (mat >> 1) * 8, k0 + (mat & 1) * 8));
    } else {
        ldsm_x4_t(b, t.addr(k0 + r8 + (mat & 1) * 8, n0 + (mat >> 1) * 8));
    }
}

// acc[NT][4] += A[m0:m0+16, k0:k0+16*KS] * B[k0:.., n0:n0+8*NT]   (one warp)
template <typename T, int NT, int KS>
__device__ __forceinline__ void warp_mma(float (*acc)[4], const Tile &A, int m0, bool a_trans, const Tile &B,
                                         int n0, bool b_trans, int k0, int lane) {
    static_assert(NT % 2 == 0, "NT must be even");
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        uint32_t a[4];
        load_a(a, A, m0, k0 + ks * 16, a_trans, lane);
#pragma unroll
        for (int nt = 0; nt < NT; nt += 2) {
            uint32_t b[4];
            load_b2(b, B, n0 + nt * 8, k0 + ks * 16, b_trans, lane);
            mma16816<T>(acc[nt], a, b[0], b[1]);
            mma16816<T>(acc[nt + 1], a, b[2], b[3]);
        }
    }
}

// Same with the A operand already in registers: af[KS][4].
template <typename T, int NT, int KS>
__device__ __forceinline__ void warp_mma_ra(float (*acc)[4], const uint32_t (*af)[4], const Tile &B, int n0,
                                            bool b_trans, int k0, int lane) {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
        for (int nt = 0; nt < NT; nt += 2) {
            uint32_t b[4];
            load_b2(b, B, n0 + nt * 8, k0 + ks * 16, b_trans, lane);
            mma16816<T>(acc[nt], af[ks], b[0], b[1]);
            mma16816<T>(acc[nt + 1], af[ks], b[2], b[3]);
        }
    }
}

template <int NT>
__device__ __forceinline__ void zero_acc(float (*acc)[4]) {
#pragma unroll
    for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
}

// Accumulators of a 16 x (16*KS) strip -> A fragments (k-steps of 16 columns).
template <typename T, int KS>
__device__ __forceinline__ void acc_to_a(uint32_t (*af)[4], const float (*acc)[4], float mul = 1.f) {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        af[ks][0] = Elt<T>::pack(acc[2 * ks][0] * mul, acc[2 * ks][1] * mul);
        af[ks][1] = Elt<T>::pack(acc[2 * ks][2] * mul, acc[2 * ks][3] * mul);
        af[ks][2] = Elt<T>::pack(acc[2 * ks + 1][0] * mul, acc[2 * ks + 1][1] * mul);
        af[ks][3] = Elt<T>::pack(acc[2 * ks + 1][2] * mul, acc[2 * ks + 1][3] * mul);
    }
}

__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(addr), "r"(v));
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint16_t lds16(uint32_t addr) {
    uint16_t v;
    asm volatile("ld.shared.b16 %0, [%1];\n" : "=h"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ void sts16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.b16 [%0], %1;\n" ::"r"(addr), "h"(v));
}

// Store a warp's 16 x (8*NT) accumulator strip (rows m0.., cols n0..) into a tile.
template <typename T, int NT>
__device__ __forceinline__ void store_acc(const Tile &t, const float (*acc)[4], int m0, int n0, int lane,
                                          float mul = 1.f) {
    const int g = lane >> 2, tq = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int col = n0 + nt * 8 + tq * 2;
        sts32(t.addr(m0 + g, col), Elt<T>::pack(acc[nt][0] * mul, acc[nt][1] * mul));
        sts32(t.addr(m0 + g + 8, col), Elt<T>::pack(acc[nt][2] * mul, acc[nt][3] * mul));
    }
}

template <typename T>
__device__ __forceinline__ float tile_get(const Tile &t, int row, int col) {
    uint16_t u = lds16(t.addr(row, col));
    T x = *reinterpret_cast<T *>(&u);
    return Elt<T>::to_f(x);
}

// ---------------------------------------------------------------- async copies

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    const int n = valid ? 16 : 0;  // 0 source bytes -> zero fill
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

// Copy `rows` (<= nrows valid) rows of `cols` 16-bit elements from global
// (row r at src + r*row_stride elements) into a tile; invalid rows are zero.
template <typename T>
__device__ __forceinline__ void load_rows_async(const Tile &t, const T *src, long long row_stride, int nrows,
                                                int valid, int cols, int tid, int nthreads) {
    const int cpr = cols / 8;
    for (int i = tid; i < nrows * cpr; i += nthreads) {
        const int r = i / cpr, c = (i % cpr) * 8;
        const bool ok = r < valid;
        const T *p = ok ? src + (long long)r * row_stride + c : src;
        cp_async16(t.addr(r, c), p, ok);
    }
}

// ---------------------------------------------------------------- chunk geometry

struct Geo {
    int B, T, Hq, Hv, N;
    int K, V;                 // head dims of the token tensors (the tiles are 128 wide; columns >= K / V are zero)
    const int32_t *cu;        // nullptr = dense
    const int32_t *cidx;      // varlen chunk table [*,2]
    const int32_t *coff;      // varlen chunk offsets [N+1]
    const int32_t *ctotal;    // varlen total chunks (< 0: the tables were not built, a malformed cu_seqlens)
    const int32_t *sorder;    // varlen sequence order, longest first (nullable): the chains' block -> sequence
    unsigned *err;            // device error word
    // Division by Hq and by the dense chunks per sequence (divisors fixed for a call) as a multiply-high, the
    // round-up method of Granlund and Montgomery ("Division by invariant integers using multiplication"):
    // n / d = (umulhi(n, m) + n) >> s for 0 <= n < 2^31, s = ceil(log2 d), m = floor(2^32 (2^s - d) / d) + 1.
    uint32_t hq_m, nt_m;
    int hq_s, nt_s;
    __device__ __forceinline__ int nt_dense() const { return (T + C - 1) / C; }
    __device__ __forceinline__ int div_hq(int n) const {
        return (int)((__umulhi((uint32_t)n, hq_m) + (uint32_t)n) >> hq_s);
    }
    __device__ __forceinline__ int div_nt(int n) const {
        return (int)((__umulhi((uint32_t)n, nt_m) + (uint32_t)n) >> nt_s);
    }
    // Sequence n: first token, length, first chunk row.  When the varlen tables were not built (the
    // chunk-table kernel latched an error) every sequence is empty, so no kernel walks a malformed range.
    __device__ __forceinline__ void seq(int n, long long &tok0, int &len, int &row0) const {
        if (cu == nullptr) {
            tok0 = (long long)n * T;
            len = T;
            row0 = n * nt_dense();
        } else if (*ctotal < 0) {
            tok0 = 0;
            len = 0;
            row0 = 0;
        } else {
            tok0 = cu[n];
            len = cu[n + 1] - cu[n];
            row0 = coff[n];
        }
    }
    // Whether chunk slot `slot` holds a chunk (the test of chunk() below, without its table reads).
    __device__ __forceinline__ bool has_chunk(int slot) const {
        return cu == nullptr ? slot < B * nt_dense() : slot < *ctotal;
    }
    // Chunk slot -> (first token, valid rows, sequence); false when past the end.
    __device__ __forceinline__ bool chunk(int slot, long long &tok0, int &len, int &n, int &ci) const {
        if (cu == nullptr) {
            const int nt = nt_dense();
            if (slot >= B * nt) return false;
            n = div_nt(slot);
            ci = slot - n * nt;
            tok0 = (long long)n * T + (long long)ci * C;
            len = min(C, T - ci * C);
            return true;
        }
        if (slot >= *ctotal) return false;
        n = cidx[2 * slot];
        ci = cidx[2 * slot + 1];
        tok0 = cu[n] + (long long)ci * C;
        len = min(C, cu[n + 1] - (int)(ci * C) - cu[n]);
        return true;
    }
};

// The multiplier and shift that divide by d (>= 1) in Geo::div_hq / div_nt.
inline void div_magic(int d, uint32_t &m, int &s) {
    if (d < 1) d = 1;  // (no division happens then: a dense call without tokens has no chunks)
    s = 0;
    while ((1ll << s) < d) ++s;
    m = (uint32_t)((((1ull << 32) * ((1ull << s) - (uint64_t)d)) / (uint64_t)d) + 1);
}

inline Geo make_geo(const Args &a) {
    Geo g;
    g.B = a.B;
    g.T = a.T;
    g.Hq = a.Hq;
    g.Hv = a.Hv;
    g.N = a.N;
    g.K = a.K;
    g.V = a.V;
    g.cu = a.cu;
    g.cidx = a.cidx;
    g.coff = a.coff;
    g.ctotal = a.ctotal;
    g.sorder = a.sorder;
    g.err = a.err;
    div_magic(a.Hq, g.hq_m, g.hq_s);
    div_magic((a.T + C - 1) / C, g.nt_m, g.nt_s);
    return g;
}

// Activations of the raw per-token gate and beta (GDR_GATE_IN_KERNEL, GDR_BETA_SIGMOID_IN_KERNEL,
// GDR_ALLOW_NEG_EIGVAL): g = logsigmoid(x) = min(x, 0) - log(1 + e^{-|x|}); beta = sigmoid(b), doubled when
// negative eigenvalues are allowed.
__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float logsigmoid_f(float x) { return fminf(x, 0.f) - log1pf(expf(-fabsf(x))); }
__device__ __forceinline__ float gate_of(float x, unsigned flags) {
    return (flags & GDR_GATE_IN_KERNEL) ? logsigmoid_f(x) : x;
}
__device__ __forceinline__ float beta_of(float b, unsigned flags) {
    if (flags & GDR_BETA_SIGMOID_IN_KERNEL) b = sigmoid_f(b);
    if (flags & GDR_ALLOW_NEG_EIGVAL) b *= 2.f;
    return b;
}

// Latch an error code in the device error word (the first code wins).
__device__ __forceinline__ void raise_error(unsigned *err, unsigned code) {
    if (err) atomicCAS(err, 0u, code);
}

}  // namespace gdr
