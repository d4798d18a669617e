/*
 * gdr.h -- C ABI of the GB300 (sm_103a) chunked Gated Delta Rule library.
 *
 * The operation (FlashQLA skill page, "Core API" and "Low-Level API"
 * sections; PR #998 "[GDN] Add FlashQLA backend dispatch", Summary):
 * for every sequence and value head j (q/k head i = j / (H_v/H_q)),
 *
 *     S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t = scale * S_t q_t
 *
 * with the state stored as h_t = S_t^T, shape [K,V] (or [V,K] when
 * GDR_STATE_V_FIRST is set).  q,k are optionally L2-normalised per token and
 * head inside the kernels (x / sqrt(sum x^2 + 1e-6)).  The library evaluates
 * it in chunks of 64 tokens (WY/UT form), on the caller's CUDA stream.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor arguments are DEVICE pointers to contiguous row-major memory
 *   allocated by the caller (the library never allocates device memory and
 *   never synchronises the stream, except gdr_get_error).  Every tensor
 *   pointer must be 16-byte aligned (GDR_ERR_ALIGN otherwise).
 * - A log-gate below -80 is taken as -80 (its factor e^g < 2e-35 already wipes
 *   the state at fp32 resolution), so g = -inf works as a hard reset; the
 *   returned g_cumsum holds the clamped sums.  NaN gates propagate.
 * - T = 0 (no tokens) is a valid problem: no step runs, the final states are
 *   the initial ones (zeros without them) and dh0 is dht (zeros without it);
 *   the token pointers may then be NULL and cu_seqlens is not read.
 * - Every launch goes to the caller's stream, and no call reads device memory
 *   on the host: the compute calls (gdr_prepare_chunks, gdr_fwd*, gdr_bwd*,
 *   gdr_decode) may be captured into a CUDA graph and replayed; gdr_get_error
 *   synchronises and may not.
 * - Dense batches: q,k [B,T,Hq,K]; v,o,do,dv [B,T,Hv,V]; g,beta,g_cumsum,
 *   dg,dbeta [B,T,Hv]; A [B,T,Hv,64]; states [B,Hv,K,V].
 *   Packed variable-length batches (cu_seqlens != NULL): the same with B = 1
 *   and T = total tokens; states are [N,Hv,K,V] for the N sequences.
 * - 8 <= K, V <= 128 and multiples of 8 (GDR_ERR_SHAPE otherwise); Hv % Hq == 0.
 *   The chunked kernels are built for K = V = 128; smaller head dims run as if
 *   zero-padded (exact: zero coordinates stay zero): the token tensors are read
 *   in place through tiles that load zeros past K / V and written clipped to
 *   them, and only the fp32 states are copied to zero-padded 128 x 128 blocks
 *   in the workspace.  They cost about what K = V = 128 costs, and the optional
 *   per-chunk states h are not offered for them (GDR_ERR_UNSUPPORTED).  The
 *   decode handles them directly.
 * - dtype (q,k,v,o,A,h,dq,dk,dv) is bf16 or fp16 (fp32 -> GDR_ERR_DTYPE);
 *   gate_dtype (g,beta,dg,dbeta) is dtype or fp32.  States, final_state,
 *   initial_state, dht, dh0 and g_cumsum are fp32.
 * - `stream` is a cudaStream_t (NULL = the legacy default stream).
 * - Calls may come from any host thread.  When the calling thread has no
 *   current CUDA context (one that has made no runtime call yet), the call
 *   makes the current device's primary context current on it (cudaSetDevice):
 *   the TMA tensor maps are encoded by a driver call that needs one.  A
 *   context the caller made current is used as it is.
 * - Every call validates its arguments on the host first and launches
 *   nothing when it returns an error.  Errors found by kernels (a malformed
 *   cu_seqlens) are latched in a device error word that gdr_get_error reads.
 *   A forward or backward whose cu_seqlens turns out malformed treats every
 *   sequence as empty: final_state = initial_state (zero without one), dh0 =
 *   dht, the other outputs unspecified; nothing outside the given buffers is
 *   touched.
 */
#ifndef GDR_H
#define GDR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdr_status {
    GDR_OK = 0,
    GDR_ERR_NULL = 1,        /* a required pointer is NULL */
    GDR_ERR_SHAPE = 2,       /* K or V not in 8..128 step 8, Hv % Hq != 0, B != 1 with cu_seqlens, negative sizes */
    GDR_ERR_DTYPE = 3,       /* fp32 or unknown q/k/v dtype, bad gate dtype */
    GDR_ERR_UNSUPPORTED = 4, /* a rejected option (multi-GPU sequence split), or an in-kernel gate
                                backward without the forward's saved buffer */
    GDR_ERR_DEVICE = 5,      /* current device is not compute capability 10.3 */
    GDR_ERR_ALIGN = 6,       /* a tensor pointer is not 16-byte aligned */
    GDR_ERR_WORKSPACE = 7,   /* workspace NULL or smaller than the size query returns */
    GDR_ERR_CUSEQLENS = 8,   /* cu_seqlens not starting at 0, decreasing, or not ending at T */
    GDR_ERR_TIMEOUT = 9,     /* a bounded device-side wait expired */
    GDR_ERR_CUDA = 10,       /* a CUDA runtime call failed (gdr_last_cuda_error names it) */
    GDR_ERR_INTERNAL = 11
} gdr_status;

typedef enum gdr_dtype { GDR_BF16 = 0, GDR_FP16 = 1, GDR_FP32 = 2 } gdr_dtype;

/* gdr_problem.flags */
#define GDR_L2NORM_QK              (1u << 0)  /* use_qk_l2norm_in_kernel */
#define GDR_STATE_V_FIRST          (1u << 1)  /* state tensors stored [..,V,K] */
/* Activations of the raw per-token scalars inside the library (the options named by
 * the FlashQLA backend's verifier, PR #998; the pages do not define them, this is the
 * library's reading):
 *   GDR_GATE_IN_KERNEL:         g holds raw gate logits x; the recurrence uses
 *                               logsigmoid(x), the log of a sigmoid decay in (0, 1)
 *   GDR_BETA_SIGMOID_IN_KERNEL: beta holds raw logits b; the recurrence uses sigmoid(b)
 *   GDR_ALLOW_NEG_EIGVAL:       beta is doubled, so the eigenvalue 1 - beta of the
 *                               transition along k spans (-1, 1)
 * g_cumsum (forward output, backward input) is the cumsum of the activated gate; dg and
 * dbeta are gradients w.r.t. the raw inputs.  The backward of GDR_GATE_IN_KERNEL needs
 * the forward's saved buffer (gdr_fwd_ex / gdr_bwd_ex), which holds the activation's
 * derivative; without it the backward returns GDR_ERR_UNSUPPORTED. */
#define GDR_GATE_IN_KERNEL         (1u << 8)
#define GDR_BETA_SIGMOID_IN_KERNEL (1u << 9)
#define GDR_ALLOW_NEG_EIGVAL       (1u << 10)
/* A sequence split across GPUs (rejected as the FlashQLA backend's verifier rejects
 * it): GDR_ERR_UNSUPPORTED. */
#define GDR_INTER_CARD_CP          (1u << 11)

#define GDR_CHUNK 64

typedef struct gdr_problem {
    int B, T;                  /* batch rows and tokens per row (packed: B = 1, T = total) */
    int Hq, Hv;                /* q/k heads and value heads, Hv % Hq == 0 */
    int K, V;                  /* head dims, 8..128 in steps of 8 (128 is the native size) */
    gdr_dtype dtype;           /* q, k, v (and o, A, h, dq, dk, dv) */
    gdr_dtype gate_dtype;      /* g, beta (and dg, dbeta): dtype or GDR_FP32 */
    float scale;               /* output scale (K^-0.5 is the usual choice) */
    const int32_t *cu_seqlens; /* DEVICE int32 [num_seqs+1] or NULL for dense */
    int num_seqs;              /* N when cu_seqlens != NULL (ignored otherwise) */
    unsigned flags;            /* GDR_* flags above */
    int num_segments;          /* intra-GPU sequence split: 0 = automatic, 1 = off,
                                  S > 1 = cut every sequence into S segments */
} gdr_problem;

/* Upper bound on the number of 64-token chunks of a problem (rows of h and of
 * chunk_indices): dense B*ceil(T/64); packed (T + N*63)/64. */
int64_t gdr_max_chunks(const gdr_problem *p);

/*
 * Varlen chunk tables (FlashQLA documentation page, utilities section:
 * prepare_lens, prepare_chunk_offsets, prepare_chunk_indices).
 *   cu_seqlens    [num_seqs+1] int32, device, in
 *   chunk_indices [max_chunks,2] int32, device, out: row r = (sequence n,
 *                 chunk c within n), ordered by n then c; rows past the total
 *                 are left untouched
 *   chunk_offsets [num_seqs+1] int32, device, out: chunks before sequence n;
 *                 chunk_offsets[num_seqs] = total
 *   total_chunks  int32 scalar, device, out
 * total_tokens (T) is used to validate cu_seqlens[num_seqs] == T; pass -1 to
 * skip that check.  A malformed cu_seqlens latches GDR_ERR_CUSEQLENS in the
 * device error word (see gdr_get_error) and writes total_chunks = 0.
 * Returns GDR_ERR_SHAPE when max_chunks is smaller than the bound
 * (total_tokens + num_seqs*(chunk_size-1)) / chunk_size.  The kernel also
 * counts the chunks before it writes anything: when they exceed max_chunks
 * (possible with total_tokens = -1) it writes nothing but total_chunks = 0 and
 * latches GDR_ERR_SHAPE in the device error word.
 */
gdr_status gdr_prepare_chunks(const int32_t *cu_seqlens, int num_seqs, int total_tokens,
                              int chunk_size, int32_t *chunk_indices, int64_t max_chunks,
                              int32_t *chunk_offsets, int32_t *total_chunks, void *stream);

/* Workspace bytes that gdr_fwd / gdr_bwd need for problem p (host-only; no
 * device access).  The workspace must be 256-byte aligned. */
gdr_status gdr_fwd_workspace_size(const gdr_problem *p, size_t *bytes);
gdr_status gdr_bwd_workspace_size(const gdr_problem *p, size_t *bytes);

/*
 * Forward (chunk_gated_delta_rule_fwd: FlashQLA skill page, "Low-Level API").
 *   in : q, k, v, g, beta (layouts above); h0 [N,Hv,K,V] fp32 or NULL (zero start)
 *   out: o [B,T,Hv,V] (dtype)
 *        final_state [N,Hv,K,V] fp32, or NULL when not wanted
 *        g_cumsum [B,T,Hv] fp32: chunk-local inclusive cumsum of g (restarting at
 *          every chunk and sequence start), or NULL
 *        A [B,T,Hv,64] (dtype): row t mod 64 of its chunk's (I + L)^-1 with
 *          L = strictly-lower(diag(beta) (k k^T o exp(G_r - G_s))), zero above the
 *          diagonal and past the sequence end, or NULL
 *        h [max_chunks,Hv,K,V] (dtype): the state before every chunk (row of chunk c
 *          of sequence n = its chunk-table row), or NULL
 *   g_cumsum and A are what gdr_bwd consumes; pass NULL for both in inference.
 * State-shaped tensors (h0, final_state, h) use [..,V,K] with GDR_STATE_V_FIRST.
 */
gdr_status gdr_fwd(const gdr_problem *p, const void *q, const void *k, const void *v,
                   const void *g, const void *beta, const float *h0, void *o, float *final_state,
                   float *g_cumsum, void *A, void *h, void *workspace, size_t workspace_bytes,
                   void *stream);

/*
 * Backward (chunk_gated_delta_rule_bwd: FlashQLA skill page, "Low-Level API";
 * the gate argument is the forward's g_cumsum, as the FlashQLA documentation
 * page's example passes the forward's returned g).
 *   in : q, k, v, g_cumsum (fp32), beta, A (from gdr_fwd), dout [B,T,Hv,V],
 *        dht [N,Hv,K,V] fp32 or NULL (zero), h0 [N,Hv,K,V] fp32 or NULL (zero)
 *   out: dq, dk [B,T,Hq,K]; dv [B,T,Hv,V] (dtype); dg, dbeta [B,T,Hv] (gate_dtype;
 *        dg is the gradient w.r.t. the raw per-token log-gate g);
 *        dh0 [N,Hv,K,V] fp32 or NULL.
 */
gdr_status gdr_bwd(const gdr_problem *p, const void *q, const void *k, const void *v,
                   const float *g_cumsum, const void *beta, const void *A, const void *dout,
                   const float *dht, const float *h0, void *dq, void *dk, void *dv, void *dg,
                   void *dbeta, float *dh0, void *workspace, size_t workspace_bytes,
                   void *stream);

/*
 * Forward and backward that hand on to the backward what it would otherwise
 * recompute (no counterpart on the pages: an addition of this library): the decayed
 * causal blocks P = scale (q^ k^T o exp(G_r - G_s)) (s <= r), the inverse q/k norms,
 * the state before every chunk and Delta = U - W h of every chunk.  The backward then
 * runs the reverse state-gradient chain alone (with the intra-GPU sequence split: the
 * reverse segment passes and that chain; the forward recompute is skipped).  Results
 * equal gdr_fwd / gdr_bwd up to rounding (the same quantities, computed by other
 * kernels).  The buffer costs memory: for B x T tokens and Hv heads about
 * B*T*Hv*(128 + 8 + 2*128*128/64 + 2*128) bytes at 16-bit data, i.e. about 0.9 KB per
 * token and head.
 *   gdr_saved_bytes: bytes of the saved buffer for problem p (host-only).
 *   saved: DEVICE buffer of at least gdr_saved_bytes bytes, 256-byte aligned, owned by
 *     the caller; NULL gives gdr_fwd / gdr_bwd exactly.  gdr_fwd_ex writes it;
 *     gdr_bwd_ex reads it and must get the buffer written by gdr_fwd_ex for the same
 *     problem, the same q, k, v, g, beta and h0 (the library cannot check this).
 *   h: must be NULL when saved is used (GDR_ERR_UNSUPPORTED otherwise): the states
 *     are then kept in the saved buffer.
 *   Other arguments, layouts and errors as gdr_fwd / gdr_bwd.
 */
gdr_status gdr_saved_bytes(const gdr_problem *p, size_t *bytes);
/* Workspace bytes that gdr_fwd_ex (backward == 0) or gdr_bwd_ex (backward != 0) needs
 * when it is given a saved buffer (host-only): the parts that the buffer holds instead
 * (P and the norms; in the backward also the states and Delta) are left out, so this is
 * at most gdr_fwd_workspace_size / gdr_bwd_workspace_size.  Errors as
 * gdr_fwd_workspace_size. */
gdr_status gdr_saved_workspace_size(const gdr_problem *p, int backward, size_t *bytes);
gdr_status gdr_fwd_ex(const gdr_problem *p, const void *q, const void *k, const void *v,
                      const void *g, const void *beta, const float *h0, void *o,
                      float *final_state, float *g_cumsum, void *A, void *h, void *workspace,
                      size_t workspace_bytes, void *saved, void *stream);
gdr_status gdr_bwd_ex(const gdr_problem *p, const void *q, const void *k, const void *v,
                      const float *g_cumsum, const void *beta, const void *A, const void *dout,
                      const float *dht, const float *h0, void *dq, void *dk, void *dv, void *dg,
                      void *dbeta, float *dh0, void *workspace, size_t workspace_bytes,
                      const void *saved, void *stream);

/*
 * Forward for callers that cannot allocate device memory (no counterpart on the
 * pages: it is an addition of this library).  Some callers may not call
 * cudaMalloc at all -- code running inside a memory pool it does not own, embedded
 * runtimes that forbid allocation after start-up, or code in a region where an
 * allocation would synchronise the device.  This entry point computes what gdr_fwd
 * computes for o and final_state (no g_cumsum, A or h outputs) but takes no
 * workspace: it uses a 64 MiB scratch array that is part of the library's device
 * image, held by every GPU that loads the library until the process exits.  It
 * allocates nothing itself and calls no allocating routine.
 *   in/out: as gdr_fwd (q, k, v, g, beta, h0 nullable; o; final_state nullable).
 *   Returns GDR_ERR_WORKSPACE when the problem's forward workspace
 *   (gdr_fwd_workspace_size) exceeds 64 MiB; every other error as gdr_fwd.
 * The first call on a device looks up the scratch array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call before
 * any stream capture.  All calls share the one array: calls whose work overlaps on
 * the GPU (different streams, or different host threads without ordering) race on
 * it and must be serialised by the caller.  Nothing in the array has to start at
 * zero; each call writes every scratch value before reading it.
 */
gdr_status gdr_fwd_noalloc(const gdr_problem *p, const void *q, const void *k, const void *v, const void *g,
                           const void *beta, const float *h0, void *o, float *final_state, void *stream);

/*
 * Recurrent decode (autoregressive inference from a cached state; the pages name
 * it in the FlashQLA skill page's inference section, whose text is cut off).  Each
 * of the T tokens of every row is applied in turn to the row's fp32 state, with
 * the recurrence the chunked forward computes in blocks: per token,
 *   S <- e^{g} S (I - beta k k^T) + beta v k^T,   o = scale S q
 * (FlashQLA skill page, "Core API"), k and q L2-normalised per token with
 * GDR_L2NORM_QK.  gdr_fwd over the same tokens gives the same o and final state up
 * to rounding.  Meant for T = 1 (one generated token) or a few tokens.
 *   in : q, k [B,T,Hq,K]; v [B,T,Hv,V]; g (the raw log-gate, as gdr_fwd's g) and
 *        beta [B,T,Hv]; state_in [B,Hv,K,V] fp32 ([B,Hv,V,K] with GDR_STATE_V_FIRST)
 *        or NULL (zero states)
 *   out: o [B,T,Hv,V] (dtype); state_out, same layout as state_in (may be state_in
 *        itself: the update runs in place).  With T = 0 only state_out is required
 *        (it receives state_in, or zeros).
 *   p: dense rows only (cu_seqlens != NULL returns GDR_ERR_UNSUPPORTED);
 *      num_segments is ignored.  Other checks and errors as gdr_fwd.
 */
gdr_status gdr_decode(const gdr_problem *p, const void *q, const void *k, const void *v, const void *g,
                      const void *beta, const float *state_in, float *state_out, void *o, void *stream);

/* Synchronises `stream`, then returns and clears the device error word of the
 * current device (GDR_OK when no kernel latched an error), or GDR_ERR_CUDA when
 * the stream reports a CUDA error. */
gdr_status gdr_get_error(void *stream);

/* Static text for a status code. */
const char *gdr_status_string(gdr_status s);

/* The name of the CUDA runtime error (e.g. "cudaErrorInvalidValue") behind the
 * calling thread's most recent GDR_ERR_CUDA, followed by the kernel whose launch
 * failed when it came from one; "cudaSuccess" before any.  The text stays valid
 * until the thread's next call that fails; the record is per host thread. */
const char *gdr_last_cuda_error(void);

/*
 * Per-kernel timing (tracing).  gdr_profile_enable(1) clears the counters and
 * from then on brackets every kernel the library launches with a pair of CUDA
 * events recorded on the launch stream (the library owns the events);
 * gdr_profile_enable(0) stops recording.  gdr_profile_read synchronises on
 * the pending events, folds them into per-kernel totals and copies up to
 * `max` entries: kernel name (static string), launch count and summed
 * milliseconds.  Returns the number of distinct kernels (may exceed max), or
 * -1 on a CUDA error.  Timing adds two event records per launch.
 */
gdr_status gdr_profile_enable(int on);
int gdr_profile_read(int max, const char **names, long long *launches, double *ms);

/*
 * Test support for the bounded device-side waits (no counterpart on the pages).
 * polls >= 0 caps the number of polls of each wait in the item loop of the
 * backward's decayed-block kernel (the one gdr_bwd / gdr_bwd_ex launch without a
 * saved buffer) at `polls`; with polls = 0 the first wait gives up without
 * looking, before its tile loads can land.  The kernel then latches
 * GDR_ERR_TIMEOUT in the device error word, lets the loads and the MMA it issued
 * finish (with its own fixed bound), frees its tensor memory and returns; the
 * results of that call are undefined.  polls < 0 restores the normal bound.
 * Process-wide setting, read by every later call.
 */
gdr_status gdr_debug_set_wait_polls(long long polls);

/* Library version, major*10000 + minor*100 + patch. */
int gdr_version(void);

#ifdef __cplusplus
}
#endif
#endif /* GDR_H */
