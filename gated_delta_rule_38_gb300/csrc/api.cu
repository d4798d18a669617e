// C-ABI entry points: argument validation, workspace layout, launch order,
// the varlen chunk-table kernel and the device error word.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "launch.h"
#include "tmap.h"

namespace gdr {

__device__ unsigned int g_gdr_error_word = 0;

// ---------------------------------------------------------------- chunk tables

// One CTA.  Validates cu_seqlens and checks that the table has room for every
// chunk (both before anything is written), then an exclusive scan of
// ceil(len/chunk) gives the offsets; each sequence's rows of the chunk table
// follow.  `order` (nullable, N entries): the sequences longest first (ties by
// index), for the chains to start the longest ones first; the identity when
// N > kOrderMax or on an error.  On an error *total = bad_total (0 for the
// public tables; -1 for the library's own, which its kernels read as "no
// tables": every sequence empty).
constexpr int kOrderMax = 2048;
__global__ void __launch_bounds__(1024) prep_chunks_kernel(const int32_t *__restrict__ cu, int N, int T, int chunk,
                                                           int32_t *__restrict__ idx, long long max_chunks,
                                                           int32_t *__restrict__ off, int32_t *__restrict__ total,
                                                           int32_t *__restrict__ order, int bad_total, unsigned *err) {
    __shared__ int s_bad;
    __shared__ int s_warp[32];
    __shared__ long long s_carry;
    __shared__ unsigned long long s_need;
    __shared__ int s_len[kOrderMax];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    if (tid == 0) {
        s_bad = (cu[0] != 0 || (T >= 0 && cu[N] != T)) ? 1 : 0;
        s_carry = 0;
        s_need = 0;
    }
    __syncthreads();
    unsigned long long need = 0;
    for (int n = tid; n < N; n += blockDim.x) {
        const int a = cu[n], b = cu[n + 1];
        if (b < a) atomicOr(&s_bad, 1);
        else need += (unsigned long long)((b - a + chunk - 1) / chunk);
    }
    if (need) atomicAdd(&s_need, need);
    __syncthreads();
    if (s_bad || (long long)s_need > max_chunks) {
        if (tid == 0) {
            *total = bad_total;
            raise_error(err, s_bad ? GDR_ERR_CUSEQLENS : GDR_ERR_SHAPE);
        }
        if (order)
            for (int n = tid; n < N; n += blockDim.x) order[n] = n;
        return;
    }
    for (int base = 0; base < N; base += blockDim.x) {
        const int n = base + tid;
        const int c = (n < N) ? (cu[n + 1] - cu[n] + chunk - 1) / chunk : 0;
        int x = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) s_warp[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = lane < nw ? s_warp[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            if (lane < nw) s_warp[lane] = w;
        }
        __syncthreads();
        const int incl = x + (warp > 0 ? s_warp[warp - 1] : 0);
        const long long excl = s_carry + incl - c;
        if (n < N) {
            off[n] = (int32_t)excl;
            for (int i = 0; i < c; ++i) {
                const long long r = excl + i;
                if (r < max_chunks) {
                    idx[2 * r] = n;
                    idx[2 * r + 1] = i;
                }
            }
        }
        __syncthreads();
        if (tid == blockDim.x - 1) s_carry += incl;
        __syncthreads();
    }
    if (tid == 0) {
        off[N] = (int32_t)s_carry;
        *total = (int32_t)s_carry;
    }
    if (order) {
        if (N > kOrderMax) {
            for (int n = tid; n < N; n += blockDim.x) order[n] = n;
            return;
        }
        for (int n = tid; n < N; n += blockDim.x) s_len[n] = cu[n + 1] - cu[n];
        __syncthreads();
        for (int n = tid; n < N; n += blockDim.x) {
            const int ln = s_len[n];
            int rank = 0;
            for (int m = 0; m < N; ++m) {
                const int lm = s_len[m];
                rank += (lm > ln || (lm == ln && m < n)) ? 1 : 0;
            }
            order[rank] = n;
        }
    }
}

cudaError_t launch_prep_chunks(const int32_t *cu, int N, int T, int chunk, int32_t *idx, int64_t max_chunks,
                               int32_t *off, int32_t *total, int32_t *order, int bad_total, unsigned *err,
                               cudaStream_t s) {
    return launch_plain(prep_chunks_kernel, dim3(1), dim3(1024), 0, s, cu, N, T, chunk, idx, (long long)max_chunks,
                        off, total, order, bad_total, err);
}

namespace {
thread_local cudaError_t g_last_cuda = cudaSuccess;  // behind this thread's latest GDR_ERR_CUDA
thread_local const char *g_last_where = nullptr;     // the launch it came from, when known
thread_local char g_last_text[160];
}  // namespace

gdr_status cuda_fail(cudaError_t e) {
    g_last_cuda = e;
    g_last_where = nullptr;
    return GDR_ERR_CUDA;
}

const char *last_cuda_error_name() {
    if (!g_last_where) return cudaGetErrorName(g_last_cuda);
    snprintf(g_last_text, sizeof(g_last_text), "%s (launching %s)", cudaGetErrorName(g_last_cuda), g_last_where);
    return g_last_text;
}

// ---------------------------------------------------------------- host helpers

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
long long g_wait_polls = -1;  // gdr_debug_set_wait_polls (< 0: every wait keeps its own bound)
int g_dev_ok[kMaxDevices];           // 0 unknown, 1 ok, 2 wrong arch
unsigned *g_err_ptr[kMaxDevices];    // device address of the error word

gdr_status device_state(unsigned **err) {
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return cuda_fail(ce);
    if (dev < 0 || dev >= kMaxDevices) return GDR_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_dev_ok[dev] == 0) {
        int major = 0, minor = 0;
        if ((ce = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (ce = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return cuda_fail(ce);
        if (major != 10 || minor != 3) {
            g_dev_ok[dev] = 2;
        } else {
            void *p = nullptr;
            if ((ce = cudaGetSymbolAddress(&p, g_gdr_error_word)) != cudaSuccess) return cuda_fail(ce);
            g_err_ptr[dev] = static_cast<unsigned *>(p);
            g_dev_ok[dev] = 1;
        }
    }
    if (g_dev_ok[dev] != 1) return GDR_ERR_DEVICE;
    if ((ce = ensure_context()) != cudaSuccess) return cuda_fail(ce);
    *err = g_err_ptr[dev];
    return GDR_OK;
}

// the gate / beta activation options
constexpr unsigned kActFlags = GDR_GATE_IN_KERNEL | GDR_BETA_SIGMOID_IN_KERNEL | GDR_ALLOW_NEG_EIGVAL;

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline size_t esize(gdr_dtype d) { return d == GDR_FP32 ? 4 : 2; }

gdr_status check_problem(const gdr_problem *p) {
    if (!p) return GDR_ERR_NULL;
    if (p->K < 8 || p->K > DK || p->K % 8 || p->V < 8 || p->V > DV || p->V % 8) return GDR_ERR_SHAPE;
    if (p->B < 1 || p->T < 0 || p->Hq < 1 || p->Hv < 1 || p->Hv % p->Hq != 0) return GDR_ERR_SHAPE;
    if (p->cu_seqlens && (p->B != 1 || p->num_seqs < 1)) return GDR_ERR_SHAPE;
    if (p->num_segments < 0) return GDR_ERR_SHAPE;
    if (p->dtype != GDR_BF16 && p->dtype != GDR_FP16) return GDR_ERR_DTYPE;
    if (p->gate_dtype != p->dtype && p->gate_dtype != GDR_FP32) return GDR_ERR_DTYPE;
    const unsigned rejected = GDR_INTER_CARD_CP;
    const unsigned known = GDR_L2NORM_QK | GDR_STATE_V_FIRST | kActFlags;
    if ((p->flags & rejected) || (p->flags & ~(known | rejected))) return GDR_ERR_UNSUPPORTED;
    return GDR_OK;
}

int num_seqs(const gdr_problem *p) { return p->cu_seqlens ? p->num_seqs : p->B; }

int64_t max_chunks_of(const gdr_problem *p) {
    if (p->cu_seqlens) return ((int64_t)p->T + (int64_t)p->num_seqs * (C - 1)) / C;
    return (int64_t)p->B * ((p->T + C - 1) / C);
}

// Segments per sequence for the intra-GPU sequence split.  Every chain CTA occupies one SM, so with
// S segments the affine passes and the full passes each run ceil(2 S streams / SMs) waves over
// ceil(chunks / S) chunks, plus a scan whose cost grows with S.  The automatic choice minimises that
// estimate against the unsplit chains; S = 1 means no split.  Host-only (the workspace size must not
// depend on the device).
constexpr int64_t kSplitSMs = 152;
int choose_nseg(const gdr_problem *p) {
    const int64_t streams = std::max<int64_t>(1, (int64_t)num_seqs(p) * p->Hv);
    const int64_t maxc = std::max<int64_t>(1, ((int64_t)p->T + C - 1) / C);
    if (p->num_segments > 0) return (int)std::max<int64_t>(1, std::min<int64_t>({p->num_segments, maxc, 64}));
    auto waves = [&](int64_t ctas) { return (ctas + kSplitSMs - 1) / kSplitSMs; };
    // Time of the forward and reverse chains in units of one step of the warp-specialised chains (one chunk
    // of one 64-column slice; every chain CTA runs alone on an SM).  Unsplit: every (sequence, head) walks
    // its chunks in two slices, in both directions.  Split into s segments: the forward's segment-affine
    // pass (two whole-width CTAs per segment and head, one per kind, 1.0 units per chunk) and full pass (two
    // slices per segment and head); the reverse zero-start pass and full pass in whole-width CTAs (one per
    // segment and head, 1.0 and 1.2 units per chunk; the reverse transfer matrices are the forward's,
    // transposed); the scans and the extra launches.
    double best = 2.0 * (double)waves(2 * streams) * (double)maxc;
    int best_s = 1;
    for (int64_t s = 2; s <= std::min<int64_t>(64, maxc); ++s) {
        const double per = (double)((maxc + s - 1) / s);
        const double w2 = (double)waves(2 * s * streams), w1 = (double)waves(s * streams);
        const double cost = per * (2.0 * w2 + 2.2 * w1) + 3.0 * (double)s + 16.0;
        if (cost < 0.95 * best) {
            best = cost;
            best_s = (int)s;
        }
    }
    return best_s;
}

struct Layout {
    size_t idx = 0, off = 0, total = 0, order = 0, gcs = 0, A = 0, P = 0, rq = 0, rk = 0, h = 0, dhn = 0, delta = 0, ddelta = 0;
    size_t geff = 0, beff = 0, dgeff = 0, dbeff = 0;  // activated gate / beta and their gradients (fp32)
    size_t seg[3] = {0, 0, 0};
    int nseg = 1;
    size_t bytes = 0;
};

// Workspace: [varlen chunk tables][fwd: g_cumsum, A scratch | bwd: states, state gradients].  With a saved
// buffer (`kept`) the parts that the buffer holds instead are left out: P and the norms in both directions,
// the states and Delta in the backward.
Layout layout_of(const gdr_problem *p, bool bwd, bool kept = false) {
    Layout L;
    size_t at = 0;
    const int64_t mc = max_chunks_of(p);
    if (p->cu_seqlens) {
        L.idx = at;
        at = round_up(at + (size_t)mc * 2 * sizeof(int32_t), 256);
        L.off = at;
        at = round_up(at + (size_t)(p->num_seqs + 1) * sizeof(int32_t), 256);
        L.total = at;
        at = round_up(at + sizeof(int32_t), 256);
        L.order = at;
        at = round_up(at + (size_t)p->num_seqs * sizeof(int32_t), 256);
    }
    const size_t tok = (size_t)p->B * p->T;
    L.nseg = choose_nseg(p);
    if (p->flags & kActFlags) {
        // fp32 activated gates for the forward; activated beta and the gradients w.r.t. the activated g and
        // beta for the backward
        const size_t sz = tok * p->Hv * sizeof(float);
        if (!bwd) {
            L.geff = at;
            at = round_up(at + sz, 256);
        }
        L.beff = at;
        at = round_up(at + sz, 256);
        if (bwd) {
            L.dgeff = at;
            at = round_up(at + sz, 256);
            L.dbeff = at;
            at = round_up(at + sz, 256);
        }
    }
    if (!bwd) {
        L.gcs = at;
        at = round_up(at + tok * p->Hv * sizeof(float), 256);
        L.A = at;
        at = round_up(at + tok * p->Hv * C * esize(p->dtype), 256);
        if (!kept) {
            // the decayed causal attention block and the inverse q/k norms for the output
            L.P = at;
            at = round_up(at + tok * p->Hv * C * esize(p->dtype), 256);
            if (p->flags & GDR_L2NORM_QK) {
                L.rq = at;
                at = round_up(at + tok * p->Hv * sizeof(float), 256);
                L.rk = at;
                at = round_up(at + tok * p->Hv * sizeof(float), 256);
            }
        }
    } else {
        const size_t st = (size_t)mc * p->Hv * DK * DV * esize(p->dtype);
        if (!kept) {
            L.h = at;
            at = round_up(at + st, 256);
        }
        L.dhn = at;
        at = round_up(at + st, 256);
        const size_t dsz = (size_t)mc * p->Hv * C * DV * esize(p->dtype);
        if (!kept) {
            L.delta = at;
            at = round_up(at + dsz, 256);
        }
        L.ddelta = at;
        at = round_up(at + dsz, 256);
        if (L.nseg == 1 && !kept) {
            L.P = at;
            at = round_up(at + tok * p->Hv * C * esize(p->dtype), 256);
            if (p->flags & GDR_L2NORM_QK) {
                L.rq = at;
                at = round_up(at + tok * p->Hv * sizeof(float), 256);
                L.rk = at;
                at = round_up(at + tok * p->Hv * sizeof(float), 256);
            }
        }
    }
    if (L.nseg > 1) {
        const size_t sz = (size_t)num_seqs(p) * p->Hv * L.nseg * DK * DV * sizeof(float);
        for (int i = 0; i < 3; ++i) {
            L.seg[i] = at;
            at = round_up(at + sz, 256);
        }
    }
    L.bytes = at;
    return L;
}

// What the forward keeps for the backward (gdr_fwd_ex / gdr_bwd_ex), 256-byte aligned parts: the decayed
// causal blocks P [tokens x Hv x 64 (dtype)], the inverse q/k norms rq, rk [tokens x Hv fp32], the states h
// and Delta of every chunk ("blocks"), with the intra-GPU split the segments' transfer matrices
// [N x Hv x segments x 128 x 128 fp32], and with GDR_GATE_IN_KERNEL first sigmoid(-x) of the raw gate
// [tokens x Hv fp32] (the derivative of the gate activation).
struct SavedLayout {
    size_t P = 0, rq = 0, rk = 0, h = 0, delta = 0, gate = 0, segp = 0, bytes = 0;
    bool blocks = false;
};
SavedLayout saved_layout_of(const gdr_problem *p) {
    SavedLayout S;
    const size_t tok = (size_t)p->B * p->T;
    size_t at = 0;
    if (p->flags & GDR_GATE_IN_KERNEL) {
        S.gate = at;
        at = round_up(at + tok * p->Hv * sizeof(float), 256);
    }
    S.blocks = true;
    const size_t mc = (size_t)max_chunks_of(p);
    S.P = at;
    at = round_up(at + tok * p->Hv * C * esize(p->dtype), 256);
    S.rq = at;
    at = round_up(at + tok * p->Hv * sizeof(float), 256);
    S.rk = at;
    at = round_up(at + tok * p->Hv * sizeof(float), 256);
    S.h = at;
    at = round_up(at + mc * p->Hv * DK * DV * esize(p->dtype), 256);
    S.delta = at;
    at = round_up(at + mc * p->Hv * C * DV * esize(p->dtype), 256);
    const int nseg = choose_nseg(p);
    if (nseg > 1) {
        // the intra-GPU split's segment transfer matrices (the identity-start affine pass of the forward)
        S.segp = at;
        at = round_up(at + (size_t)num_seqs(p) * p->Hv * nseg * DK * DV * sizeof(float), 256);
    }
    S.bytes = at;
    return S;
}

// Head dimensions below 128 run through the K = V = 128 path: the kernels read the token tensors through TMA
// boxes that load zeros past K / V (so their 128-wide tiles see zero-padded rows) and clip their stores there;
// the fp32 states, which the kernels address directly, are copied to and from zero-padded 128 x 128 blocks
// (pad.cu).  Zero padding is exact for this recurrence (pad.cu).
bool is_padded(const gdr_problem *p) { return p->K != DK || p->V != DV; }
gdr_problem padded_problem(const gdr_problem *p) {
    gdr_problem q = *p;
    q.K = DK;
    q.V = DV;
    return q;
}
// Workspace of a call with small head dims: [padded states][the K = V = 128 call's own workspace].
struct PadLayout {
    size_t h0 = 0, fin = 0, dht = 0, dh0 = 0;
    size_t inner = 0, bytes = 0;
};
PadLayout pad_layout_of(const gdr_problem *p, bool bwd, bool kept) {
    PadLayout P;
    const size_t st = (size_t)num_seqs(p) * p->Hv * DK * DV * sizeof(float);
    size_t at = 0;
    auto take = [&](size_t &off, size_t n) {
        off = at;
        at = round_up(at + n, 256);
    };
    take(P.h0, st);
    if (!bwd) {
        take(P.fin, st);
    } else {
        take(P.dht, st);
        take(P.dh0, st);
    }
    P.inner = at;
    const gdr_problem p128 = padded_problem(p);
    P.bytes = at + layout_of(&p128, bwd, kept).bytes;
    return P;
}

SegWs seg_ws(const Layout &L, char *ws) {
    SegWs sw;
    sw.nseg = L.nseg;
    sw.start = L.nseg > 1 ? reinterpret_cast<float *>(ws + L.seg[0]) : nullptr;
    sw.end0 = L.nseg > 1 ? reinterpret_cast<float *>(ws + L.seg[1]) : nullptr;
    sw.end1 = L.nseg > 1 ? reinterpret_cast<float *>(ws + L.seg[2]) : nullptr;
    return sw;
}

Args make_args(const gdr_problem *p, unsigned *err) {
    Args a;
    a.B = p->B;
    a.T = p->T;
    a.Hq = p->Hq;
    a.Hv = p->Hv;
    a.K = p->K;
    a.V = p->V;
    a.N = num_seqs(p);
    a.bf16 = p->dtype == GDR_BF16;
    a.gate_f32 = p->gate_dtype == GDR_FP32;
    a.l2norm = (p->flags & GDR_L2NORM_QK) != 0;
    a.v_first = (p->flags & GDR_STATE_V_FIRST) != 0;
    a.scale = p->scale;
    a.cu = p->cu_seqlens;
    a.cidx = a.coff = a.ctotal = a.sorder = nullptr;
    a.max_chunks = max_chunks_of(p);
    a.err = err;
    a.flags = p->flags;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        a.wait_polls = g_wait_polls;
    }
    return a;
}

gdr_status check_ws(const Layout &L, void *ws, size_t bytes) {
    if (L.bytes == 0) return GDR_OK;
    if (!ws || bytes < L.bytes) return GDR_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return GDR_ERR_ALIGN;
    return GDR_OK;
}

gdr_status cuda_status(cudaError_t e) { return e == cudaSuccess ? GDR_OK : cuda_fail(e); }

// ---- per-kernel timing: event pairs recorded around each launch while enabled
enum KernelId {
    K_PREP = 0, K_WY_FWD, K_CHAIN_FWD, K_CHAIN_FWD_RECOMPUTE, K_CHAIN_BWD, K_CHAIN_PAIR, K_BWD_CHUNK, K_CHUNK_P,
    K_CHAIN_REV, K_GATE_ACT, K_PAD, K_ONECHUNK, K_COUNT
};
const char *const kKernelNames[K_COUNT] = {"prep_chunks", "wy_fwd",     "chain_fwd", "chain_fwd_recompute",
                                           "chain_bwd",   "chain_pair", "bwd_chunk", "chunk_p",
                                           "chain_rev",   "gate_act",   "pad",       "onechunk_dg"};
struct Pending {
    int id;
    cudaEvent_t a, b;
};
struct Profiler {
    std::mutex mu;
    bool on = false;
    std::vector<Pending> pending;
    std::vector<cudaEvent_t> pool;
    double ms[K_COUNT] = {};
    long long count[K_COUNT] = {};
} g_prof;

cudaEvent_t prof_event() {
    if (!g_prof.pool.empty()) {
        cudaEvent_t e = g_prof.pool.back();
        g_prof.pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// Launch through f, bracketed by events when profiling is on.
template <typename F>
gdr_status timed(int id, cudaStream_t s, F &&f) {
    cudaEvent_t a = nullptr, b = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_prof.mu);
        if (g_prof.on) {
            a = prof_event();
            b = prof_event();
        }
    }
    if (a) cudaEventRecord(a, s);
    const cudaError_t e = f();
    if (b) {
        cudaEventRecord(b, s);
        std::lock_guard<std::mutex> lk(g_prof.mu);
        g_prof.pending.push_back(Pending{id, a, b});
    }
    const gdr_status st = cuda_status(e);
    if (st != GDR_OK) g_last_where = kKernelNames[id];
    return st;
}

// Build the varlen chunk tables in the workspace (no-op for dense batches).
gdr_status tables(const gdr_problem *p, Args &a, char *ws, const Layout &L, cudaStream_t s) {
    if (!p->cu_seqlens) return GDR_OK;
    a.cidx = reinterpret_cast<int32_t *>(ws + L.idx);
    a.coff = reinterpret_cast<int32_t *>(ws + L.off);
    a.ctotal = reinterpret_cast<int32_t *>(ws + L.total);
    a.sorder = reinterpret_cast<int32_t *>(ws + L.order);
    return timed(K_PREP, s, [&] {
        return launch_prep_chunks(p->cu_seqlens, p->num_seqs, p->T, C, const_cast<int32_t *>(a.cidx), a.max_chunks,
                                  const_cast<int32_t *>(a.coff), const_cast<int32_t *>(a.ctotal),
                                  const_cast<int32_t *>(a.sorder), -1, a.err, s);
    });
}

}  // namespace
}  // namespace gdr

using namespace gdr;

extern "C" {

int64_t gdr_max_chunks(const gdr_problem *p) {
    if (check_problem(p) != GDR_OK) return -1;
    return max_chunks_of(p);
}

gdr_status gdr_prepare_chunks(const int32_t *cu_seqlens, int num_seqs, int total_tokens, int chunk_size,
                              int32_t *chunk_indices, int64_t max_chunks, int32_t *chunk_offsets,
                              int32_t *total_chunks, void *stream) {
    if (!cu_seqlens || !chunk_indices || !chunk_offsets || !total_chunks) return GDR_ERR_NULL;
    if (num_seqs < 1 || chunk_size < 1 || total_tokens < -1) return GDR_ERR_SHAPE;
    if (total_tokens >= 0) {
        const int64_t bound = ((int64_t)total_tokens + (int64_t)num_seqs * (chunk_size - 1)) / chunk_size;
        if (max_chunks < bound) return GDR_ERR_SHAPE;
    }
    unsigned *err = nullptr;
    gdr_status st = device_state(&err);
    if (st != GDR_OK) return st;
    return cuda_status(launch_prep_chunks(cu_seqlens, num_seqs, total_tokens, chunk_size, chunk_indices,
                                          max_chunks, chunk_offsets, total_chunks, nullptr, 0, err,
                                          static_cast<cudaStream_t>(stream)));
}

gdr_status gdr_fwd_workspace_size(const gdr_problem *p, size_t *bytes) {
    gdr_status st = check_problem(p);
    if (st != GDR_OK) return st;
    if (!bytes) return GDR_ERR_NULL;
    *bytes = is_padded(p) ? pad_layout_of(p, false, false).bytes : layout_of(p, false).bytes;
    return GDR_OK;
}

gdr_status gdr_bwd_workspace_size(const gdr_problem *p, size_t *bytes) {
    gdr_status st = check_problem(p);
    if (st != GDR_OK) return st;
    if (!bytes) return GDR_ERR_NULL;
    *bytes = is_padded(p) ? pad_layout_of(p, true, false).bytes : layout_of(p, true).bytes;
    return GDR_OK;
}

gdr_status gdr_saved_workspace_size(const gdr_problem *p, int backward, size_t *bytes) {
    gdr_status st = check_problem(p);
    if (st != GDR_OK) return st;
    if (!bytes) return GDR_ERR_NULL;
    *bytes = is_padded(p) ? pad_layout_of(p, backward != 0, true).bytes : layout_of(p, backward != 0, true).bytes;
    return GDR_OK;
}

gdr_status gdr_saved_bytes(const gdr_problem *p, size_t *bytes) {
    if (!bytes) return GDR_ERR_NULL;
    gdr_status st = check_problem(p);
    if (st != GDR_OK) return st;
    const gdr_problem p128 = padded_problem(p);
    *bytes = saved_layout_of(&p128).bytes;
    return GDR_OK;
}

gdr_status gdr_fwd(const gdr_problem *p, const void *q, const void *k, const void *v, const void *g,
                   const void *beta, const float *h0, void *o, float *final_state, float *g_cumsum, void *A,
                   void *h, void *workspace, size_t workspace_bytes, void *stream) {
    return gdr_fwd_ex(p, q, k, v, g, beta, h0, o, final_state, g_cumsum, A, h, workspace, workspace_bytes, nullptr,
                      stream);
}

static gdr_status fwd_core(const gdr_problem *p, int tk, int tv, const void *q, const void *k, const void *v,
                           const void *g, const void *beta, const float *h0, void *o, float *final_state,
                           float *g_cumsum, void *A, void *h, void *workspace, size_t workspace_bytes, void *saved,
                           void *stream);
static gdr_status bwd_core(const gdr_problem *p, int tk, int tv, const void *q, const void *k, const void *v,
                           const float *g_cumsum, const void *beta, const void *A, const void *dout, const float *dht,
                           const float *h0, void *dq, void *dk, void *dv, void *dg, void *dbeta, float *dh0,
                           void *workspace, size_t workspace_bytes, const void *saved, void *stream);

// A problem with no tokens (T = 0) runs no step of the recurrence: the state passes through unchanged (the
// final states are the initial ones, the initial states' gradient is the final states'; zeros where the
// source is absent).  Nothing else is read or written, so the token pointers may be NULL; cu_seqlens is not
// read.
static gdr_status no_tokens(const gdr_problem *p, const float *src, float *dst, void *stream) {
    if (src && !aligned16(src)) return GDR_ERR_ALIGN;
    if (!dst) return GDR_OK;
    if (!aligned16(dst)) return GDR_ERR_ALIGN;
    unsigned *err = nullptr;
    gdr_status st = device_state(&err);
    if (st != GDR_OK) return st;
    const size_t bytes = (size_t)num_seqs(p) * p->Hv * p->K * p->V * sizeof(float);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return cuda_status(src ? cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s)
                           : cudaMemsetAsync(dst, 0, bytes, s));
}

gdr_status gdr_fwd_ex(const gdr_problem *p, const void *q, const void *k, const void *v, const void *g,
                      const void *beta, const float *h0, void *o, float *final_state, float *g_cumsum, void *A,
                      void *h, void *workspace, size_t workspace_bytes, void *saved, void *stream) {
    gdr_status st = check_problem(p);
    if (st != GDR_OK) return st;
    if (p->T == 0) return no_tokens(p, h0, final_state, stream);
    if (!q || !k || !v || !g || !beta || !o) return GDR_ERR_NULL;
    const void *ptrs[] = {q, k, v, g, beta, h0, o, final_state, g_cumsum, A, h, p->cu_seqlens, saved};
    for (const void *x : ptrs)
        if (x && !aligned16(x)) return GDR_ERR_ALIGN;
    if (is_padded(p)) {
        // the K = V = 128 path on the caller's token tensors, with zero-padded states (the per-chunk states h
        // are not offered here)
        if (h) return GDR_ERR_UNSUPPORTED;
        const PadLayout P = pad_layout_of(p, false, saved != nullptr);
        if (!workspace || workspace_bytes < P.bytes) return GDR_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(workspace) & 255u) return GDR_ERR_ALIGN;
        unsigned *err = nullptr;
        if ((st = device_state(&err)) != GDR_OK) return st;
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        char *ws = static_cast<char *>(workspace);
        const long long nh = (long long)num_seqs(p) * p->Hv;
        const bool vf = (p->flags & GDR_STATE_V_FIRST) != 0;
        const int R = vf ? p->V : p->K, Cc = vf ? p->K : p->V;
        if (h0 && (st = timed(K_PAD, s, [&] {
                       return launch_pad_state(h0, reinterpret_cast<float *>(ws + P.h0), nh, R, Cc, s);
                   })) != GDR_OK)
            return st;
        const gdr_problem p128 = padded_problem(p);
        if ((st = fwd_core(&p128, p->K, p->V, q, k, v, g, beta, h0 ? reinterpret_cast<const float *>(ws + P.h0) : nullptr,
                           o, final_state ? reinterpret_cast<float *>(ws + P.fin) : nullptr, g_cumsum, A, nullptr,
                           ws + P.inner, workspace_bytes - P.inner, saved, stream)) != GDR_OK)
            return st;
        if (!final_state) return GDR_OK;
        return timed(K_PAD, s, [&] {
            return launch_unpad_state(reinterpret_cast<const float *>(ws + P.fin), final_state, nh, R, Cc, s);
        });
    }
    return fwd_core(p, p->K, p->V, q, k, v, g, beta, h0, o, final_state, g_cumsum, A, h, workspace, workspace_bytes,
                    saved, stream);
}

// The K = V = 128 forward; tk, tv: the head dims of the token tensors (below 128 they are read through boxes that
// load zeros past them, and o is stored clipped to tv columns).
static gdr_status fwd_core(const gdr_problem *p, int tk, int tv, const void *q, const void *k, const void *v,
                           const void *g, const void *beta, const float *h0, void *o, float *final_state,
                           float *g_cumsum, void *A, void *h, void *workspace, size_t workspace_bytes, void *saved,
                           void *stream) {
    gdr_status st;
    // with a saved buffer the states go there (one copy of them per call)
    if (h && saved && saved_layout_of(p).blocks) return GDR_ERR_UNSUPPORTED;
    const Layout L = layout_of(p, false, saved != nullptr);
    if ((st = check_ws(L, workspace, workspace_bytes)) != GDR_OK) return st;
    unsigned *err = nullptr;
    if ((st = device_state(&err)) != GDR_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    Args a = make_args(p, err);
    a.K = tk;
    a.V = tv;
    if ((st = tables(p, a, ws, L, s)) != GDR_OK) return st;
    const SavedLayout S = saved_layout_of(p);
    if (p->flags & kActFlags) {
        // the activated gate and beta (fp32) replace the raw ones for the rest of the pass
        float *ge = reinterpret_cast<float *>(ws + L.geff), *be = reinterpret_cast<float *>(ws + L.beff);
        float *sg = (saved && (p->flags & GDR_GATE_IN_KERNEL)) ? reinterpret_cast<float *>(static_cast<char *>(saved) + S.gate)
                                                                : nullptr;
        if ((st = timed(K_GATE_ACT, s, [&] { return launch_gate_act_fwd(a, g, beta, p->flags, ge, be, sg, s); })) != GDR_OK)
            return st;
        g = ge;
        beta = be;
        a.gate_f32 = true;
    }
    float *gcs = g_cumsum ? g_cumsum : reinterpret_cast<float *>(ws + L.gcs);
    void *Aw = A ? A : static_cast<void *>(ws + L.A);
    SegWs sw = seg_ws(L, ws);
    // P and the norms go to the caller's saved buffer when one is given (the backward then skips its P pass)
    char *sv = (saved && S.blocks) ? static_cast<char *>(saved) : nullptr;
    // ... and so do the split's segment transfer matrices (the backward's transfer matrices are their transposes)
    if (sv && sw.nseg > 1) sw.end1 = reinterpret_cast<float *>(sv + S.segp);
    void *Pw = sv ? sv + S.P : ws + L.P;
    float *rqw = a.l2norm ? reinterpret_cast<float *>(sv ? sv + S.rq : ws + L.rq) : nullptr;
    float *rkw = a.l2norm ? reinterpret_cast<float *>(sv ? sv + S.rk : ws + L.rk) : nullptr;
    // ... and the state before every chunk and Delta of every chunk (the backward then runs no forward recompute)
    void *hs = sv ? static_cast<void *>(sv + S.h) : h;
    void *dls = sv ? static_cast<void *>(sv + S.delta) : nullptr;
    if ((st = timed(K_WY_FWD, s, [&] { return launch_wy_fwd(a, q, k, g, beta, gcs, Aw, Pw, rqw, rkw, s); })) !=
        GDR_OK)
        return st;
    // the intra-GPU split: the segment-affine passes and the scan give every segment's start state, then the
    // same warp-specialised recurrence runs every segment from its start
    return timed(K_CHAIN_FWD, s, [&] {
        if (sw.nseg > 1) {
            cudaError_t e = launch_chain_ws_affine(a, q, k, v, gcs, beta, Aw, rqw, rkw, sw.nseg, sw.end0, sw.end1, s);
            if (e == cudaSuccess) e = launch_fwd_compose(a, h0, sw, s);
            if (e != cudaSuccess) return e;
        }
        return launch_chain_ws(a, q, k, v, gcs, beta, Aw, Pw, rqw, rkw, h0, sw.nseg > 1 ? sw.start : nullptr, sw.nseg,
                               o, final_state, hs, sv ? false : a.v_first, dls, s);
    });
}

gdr_status gdr_bwd(const gdr_problem *p, const void *q, const void *k, const void *v, const float *g_cumsum,
                   const void *beta, const void *A, const void *dout, const float *dht, const float *h0, void *dq,
                   void *dk, void *dv, void *dg, void *dbeta, float *dh0, void *workspace, size_t workspace_bytes,
                   void *stream) {
    return gdr_bwd_ex(p, q, k, v, g_cumsum, beta, A, dout, dht, h0, dq, dk, dv, dg, dbeta, dh0, workspace,
                      workspace_bytes, nullptr, stream);
}

gdr_status gdr_bwd_ex(const gdr_problem *p, const void *q, const void *k, const void *v, const float *g_cumsum,
                      const void *beta, const void *A, const void *dout, const float *dht, const float *h0, void *dq,
                      void *dk, void *dv, void *dg, void *dbeta, float *dh0, void *workspace,
                      size_t workspace_bytes, const void *saved, void *stream) {
    gdr_status st = check_problem(p);
    if (st != GDR_OK) return st;
    if (p->T == 0) return no_tokens(p, dht, dh0, stream);
    if (!q || !k || !v || !g_cumsum || !beta || !A || !dout || !dq || !dk || !dv || !dg || !dbeta)
        return GDR_ERR_NULL;
    const void *ptrs[] = {q, k, v, g_cumsum, beta, A, dout, dht, h0, dq, dk, dv, dg, dbeta, dh0, p->cu_seqlens, saved};
    for (const void *x : ptrs)
        if (x && !aligned16(x)) return GDR_ERR_ALIGN;
    // the gate activation's derivative comes from the forward's saved buffer
    if ((p->flags & GDR_GATE_IN_KERNEL) && !saved) return GDR_ERR_UNSUPPORTED;
    if (is_padded(p)) {
        // the K = V = 128 path on the caller's token tensors, with zero-padded states
        const PadLayout P = pad_layout_of(p, true, saved != nullptr);
        if (!workspace || workspace_bytes < P.bytes) return GDR_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(workspace) & 255u) return GDR_ERR_ALIGN;
        unsigned *err = nullptr;
        if ((st = device_state(&err)) != GDR_OK) return st;
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        char *ws = static_cast<char *>(workspace);
        const long long nh = (long long)num_seqs(p) * p->Hv;
        const bool vf = (p->flags & GDR_STATE_V_FIRST) != 0;
        const int R = vf ? p->V : p->K, Cc = vf ? p->K : p->V;
        if ((h0 || dht) && (st = timed(K_PAD, s, [&] {
                                cudaError_t e = cudaSuccess;
                                if (h0) e = launch_pad_state(h0, reinterpret_cast<float *>(ws + P.h0), nh, R, Cc, s);
                                if (e == cudaSuccess && dht)
                                    e = launch_pad_state(dht, reinterpret_cast<float *>(ws + P.dht), nh, R, Cc, s);
                                return e;
                            })) != GDR_OK)
            return st;
        const gdr_problem p128 = padded_problem(p);
        if ((st = bwd_core(&p128, p->K, p->V, q, k, v, g_cumsum, beta, A, dout,
                           dht ? reinterpret_cast<const float *>(ws + P.dht) : nullptr,
                           h0 ? reinterpret_cast<const float *>(ws + P.h0) : nullptr, dq, dk, dv, dg, dbeta,
                           dh0 ? reinterpret_cast<float *>(ws + P.dh0) : nullptr, ws + P.inner,
                           workspace_bytes - P.inner, saved, stream)) != GDR_OK)
            return st;
        if (!dh0) return GDR_OK;
        return timed(K_PAD, s, [&] {
            return launch_unpad_state(reinterpret_cast<const float *>(ws + P.dh0), dh0, nh, R, Cc, s);
        });
    }
    return bwd_core(p, p->K, p->V, q, k, v, g_cumsum, beta, A, dout, dht, h0, dq, dk, dv, dg, dbeta, dh0, workspace,
                    workspace_bytes, saved, stream);
}

// The K = V = 128 backward; tk, tv: the head dims of the token tensors (below 128 they are read through boxes that
// load zeros past them, and dq, dk, dv are stored clipped to them).
static gdr_status bwd_core(const gdr_problem *p, int tk, int tv, const void *q, const void *k, const void *v,
                           const float *g_cumsum, const void *beta, const void *A, const void *dout, const float *dht,
                           const float *h0, void *dq, void *dk, void *dv, void *dg, void *dbeta, float *dh0,
                           void *workspace, size_t workspace_bytes, const void *saved, void *stream) {
    gdr_status st;
    const Layout L = layout_of(p, true, saved != nullptr);
    if ((st = check_ws(L, workspace, workspace_bytes)) != GDR_OK) return st;
    unsigned *err = nullptr;
    if ((st = device_state(&err)) != GDR_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    Args a = make_args(p, err);
    a.K = tk;
    a.V = tv;
    if ((st = tables(p, a, ws, L, s)) != GDR_OK) return st;
    const Args a_raw = a;
    const SavedLayout S = saved_layout_of(p);
    void *dg_out = dg, *dbeta_out = dbeta;
    const void *beta_raw = beta;
    if (p->flags & kActFlags) {
        // the pass runs on the activated beta and yields the gradients w.r.t. the activated g and beta (fp32)
        float *be = reinterpret_cast<float *>(ws + L.beff);
        if ((st = timed(K_GATE_ACT, s, [&] { return launch_gate_act_beta(a, beta, p->flags, be, s); })) != GDR_OK)
            return st;
        beta = be;
        dg = ws + L.dgeff;
        dbeta = ws + L.dbeff;
        a.gate_f32 = true;
    }
    void *hw = ws + L.h, *dhw = ws + L.dhn, *dlw = ws + L.delta, *ddlw = ws + L.ddelta;
    // states and Delta of every chunk (the forward's, or recomputed), the reverse state-gradient chain, then
    // every chunk's gradients in parallel
    const SegWs sw = seg_ws(L, ws);
    const char *sv = (saved && S.blocks) ? static_cast<const char *>(saved) : nullptr;
    if (sv) {
        // the states, Delta, P and the norms are the forward's: the reverse chain alone, in 64-column slices
        // (with the intra-GPU split: after the reverse segment-affine passes and the scan, every segment from
        // the gradient at its end)
        void *Pw = const_cast<char *>(sv + S.P);
        float *rqw = a.l2norm ? reinterpret_cast<float *>(const_cast<char *>(sv + S.rq)) : nullptr;
        float *rkw = a.l2norm ? reinterpret_cast<float *>(const_cast<char *>(sv + S.rk)) : nullptr;
        hw = const_cast<char *>(sv + S.h);
        dlw = const_cast<char *>(sv + S.delta);
        if ((st = timed(sw.nseg > 1 ? K_CHAIN_BWD : K_CHAIN_REV, s, [&] {
                 if (sw.nseg > 1) {
                     // the split: every segment's gradient at its start from a zero end (the same reverse chain,
                     // no per-chunk outputs), then the scan with the forward's transfer matrices, transposed
                     cudaError_t e = launch_chain_rev(a, q, k, g_cumsum, beta, A, Pw, rqw, rkw, dout, nullptr, nullptr,
                                                      sw.nseg, nullptr, nullptr, nullptr, sw.end0, s);
                     if (e == cudaSuccess)
                         e = launch_rev_compose(a, dht, reinterpret_cast<const float *>(sv + S.segp), sw, s);
                     if (e != cudaSuccess) return e;
                 }
                 return launch_chain_rev(a, q, k, g_cumsum, beta, A, Pw, rqw, rkw, dout, dht,
                                         sw.nseg > 1 ? sw.start : nullptr, sw.nseg, dhw, ddlw, dh0, nullptr, s);
             })) != GDR_OK)
            return st;
    } else if (sw.nseg == 1) {
        // P and the norms recomputed from g_cumsum
        void *Pw = ws + L.P;
        float *rqw = a.l2norm ? reinterpret_cast<float *>(ws + L.rq) : nullptr;
        float *rkw = a.l2norm ? reinterpret_cast<float *>(ws + L.rk) : nullptr;
        if ((st = timed(K_CHUNK_P, s, [&] { return launch_chunk_p_tc(a, q, k, g_cumsum, Pw, rqw, rkw, s); })) != GDR_OK)
            return st;
        if ((st = timed(K_CHAIN_PAIR, s, [&] {
                 return launch_chain_ws_pair(a, q, k, v, g_cumsum, beta, A, Pw, rqw, rkw, h0, hw, dlw, dout, dht, dhw,
                                             ddlw, dh0, s);
             })) != GDR_OK)
            return st;
    } else if ((st = timed(K_CHAIN_FWD_RECOMPUTE, s, [&] {
             return launch_chain_fwd(a, q, k, v, g_cumsum, beta, A, h0, nullptr, nullptr, hw, false, dlw, sw, s);
         })) != GDR_OK) {
        return st;
    } else if ((st = timed(K_CHAIN_BWD, s, [&] {
                    return launch_chain_bwd(a, q, k, g_cumsum, beta, A, dout, dht, dhw, ddlw, dh0, sw, s);
                })) != GDR_OK) {
        return st;
    }
    if ((st = timed(K_BWD_CHUNK, s, [&] {
             return launch_bwd_chunk_tc(a, q, k, v, g_cumsum, beta, A, dout, hw, dhw, dlw, ddlw, dq, dk, dv, dg, dbeta,
                                        s);
         })) != GDR_OK)
        return st;
    // sequences of one chunk with both states: the exact <dht, h0> in their dg (possible only in packed batches
    // or when T <= 64)
    if (h0 && dht && (p->cu_seqlens || p->T <= C) &&
        (st = timed(K_ONECHUNK, s, [&] { return launch_onechunk_dg(a, h0, dht, g_cumsum, dg, s); })) != GDR_OK)
        return st;
    if (!(p->flags & kActFlags)) return GDR_OK;
    // gradients w.r.t. the raw gate and beta
    const float *sg = (p->flags & GDR_GATE_IN_KERNEL)
                          ? reinterpret_cast<const float *>(static_cast<const char *>(saved) + S.gate)
                          : nullptr;
    return timed(K_GATE_ACT, s, [&] {
        return launch_gate_act_bwd(a_raw, static_cast<const float *>(dg), static_cast<const float *>(dbeta), sg,
                                   beta_raw, p->flags, dg_out, dbeta_out, s);
    });
}

gdr_status gdr_decode(const gdr_problem *p, const void *q, const void *k, const void *v, const void *g,
                      const void *beta, const float *state_in, float *state_out, void *o, void *stream) {
    gdr_status st = check_problem(p);
    if (st != GDR_OK) return st;
    if (p->cu_seqlens) return GDR_ERR_UNSUPPORTED;  // dense rows only (each row its own cached state)
    if ((long long)p->B * p->Hv > 0x7fffffffLL) return GDR_ERR_SHAPE;  // one block per (row, head)
    if (!state_out || (p->T > 0 && (!q || !k || !v || !g || !beta || !o))) return GDR_ERR_NULL;
    const void *ptrs[] = {q, k, v, g, beta, state_in, state_out, o};
    for (const void *x : ptrs)
        if (x && !aligned16(x)) return GDR_ERR_ALIGN;
    unsigned *err = nullptr;
    if ((st = device_state(&err)) != GDR_OK) return st;
    const Args a = make_args(p, err);
    return cuda_status(launch_decode(a, q, k, v, g, beta, state_in, state_out, o, static_cast<cudaStream_t>(stream)));
}

gdr_status gdr_get_error(void *stream) {
    unsigned *err = nullptr;
    gdr_status st = device_state(&err);
    if (st != GDR_OK) return st;
    cudaError_t ce = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (ce != cudaSuccess) return cuda_fail(ce);
    unsigned code = 0;
    if ((ce = cudaMemcpy(&code, err, sizeof(code), cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(ce);
    const unsigned zero = 0;
    if (code != 0 && cudaMemcpy(err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
        return GDR_ERR_CUDA;
    return static_cast<gdr_status>(code);
}

const char *gdr_status_string(gdr_status s) {
    switch (s) {
        case GDR_OK: return "ok";
        case GDR_ERR_NULL: return "a required pointer is NULL";
        case GDR_ERR_SHAPE: return "unsupported shape (K and V multiples of 8 in [8, 128], Hv % Hq == 0, B == 1 with cu_seqlens)";
        case GDR_ERR_DTYPE: return "unsupported dtype (q/k/v must be bf16 or fp16; gates the same or fp32)";
        case GDR_ERR_UNSUPPORTED: return "unsupported option";
        case GDR_ERR_DEVICE: return "the current device is not compute capability 10.3 (sm_103a)";
        case GDR_ERR_ALIGN: return "a tensor pointer is not 16-byte aligned (workspace: 256-byte)";
        case GDR_ERR_WORKSPACE: return "workspace missing or too small";
        case GDR_ERR_CUSEQLENS: return "malformed cu_seqlens";
        case GDR_ERR_TIMEOUT: return "a bounded device-side wait expired";
        case GDR_ERR_CUDA: return "CUDA runtime error";
        case GDR_ERR_INTERNAL: return "internal error";
    }
    return "unknown status";
}

const char *gdr_last_cuda_error(void) { return gdr::last_cuda_error_name(); }

int gdr_version(void) { return 100; }

gdr_status gdr_debug_set_wait_polls(long long polls) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_wait_polls = polls < 0 ? -1 : polls;
    return GDR_OK;
}

gdr_status gdr_profile_enable(int on) {
    std::lock_guard<std::mutex> lk(g_prof.mu);
    if (on) {
        for (int i = 0; i < K_COUNT; ++i) {
            g_prof.ms[i] = 0.0;
            g_prof.count[i] = 0;
        }
    }
    g_prof.on = on != 0;
    return GDR_OK;
}

int gdr_profile_read(int max, const char **names, long long *launches, double *ms) {
    std::lock_guard<std::mutex> lk(g_prof.mu);
    int rc = 0;
    for (const Pending &pd : g_prof.pending) {
        float t = 0.f;
        if (cudaEventSynchronize(pd.b) != cudaSuccess || cudaEventElapsedTime(&t, pd.a, pd.b) != cudaSuccess) rc = -1;
        g_prof.ms[pd.id] += t;
        g_prof.count[pd.id] += 1;
        g_prof.pool.push_back(pd.a);
        g_prof.pool.push_back(pd.b);
    }
    g_prof.pending.clear();
    if (rc < 0) return -1;
    int n = 0;
    for (int i = 0; i < K_COUNT; ++i) {
        if (g_prof.count[i] == 0) continue;
        if (n < max) {
            if (names) names[n] = kKernelNames[i];
            if (launches) launches[n] = g_prof.count[i];
            if (ms) ms[n] = g_prof.ms[i];
        }
        ++n;
    }
    return n;
}

}  // extern "C"
