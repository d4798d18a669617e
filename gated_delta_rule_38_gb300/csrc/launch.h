// Host-side launchers shared between the translation units of the library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gdr.h"

namespace gdr {

// Everything a kernel needs to address one problem's tensors.
struct Args {
    int B, T, Hq, Hv, N;
    int K, V;         // head dims of the token tensors (the chunked kernels' tiles are 128 wide and load zeros past
                      // them; the decode takes any <= 128)
    bool bf16;        // element type of q,k,v,... (else fp16)
    bool gate_f32;    // g, beta (dg, dbeta) are fp32
    bool l2norm;
    bool v_first;
    float scale;
    const int32_t *cu;       // device cu_seqlens or nullptr
    const int32_t *cidx;     // device chunk table [max_chunks,2] (varlen)
    const int32_t *coff;     // device chunk offsets [N+1] (varlen)
    const int32_t *ctotal;   // device total chunks (varlen)
    const int32_t *sorder;   // device sequence order, longest first (varlen; nullable)
    int64_t max_chunks;
    unsigned *err;           // device error word
    long long wait_polls;    // >= 0: poll budget of the waits that honour it (test support); < 0 = default
    unsigned flags;          // the problem's GDR_* flags
};

// Workspace of the intra-GPU sequence split (nseg segments per sequence; nseg == 1: no split):
// three [N,Hv,nseg,128,128] fp32 arrays of transposed states.
struct SegWs {
    int nseg;
    float *start, *end0, *end1;
};

// Launch with programmatic stream serialisation: the kernel may begin launching while the previous kernel in
// the stream finishes (its blocks then wait in griddep_wait, before any global memory access, until that
// kernel is complete), which hides the launch gap between the step's kernels.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Launch on stream s and return the launch's own status: not the calling thread's last runtime error, which
// can hold an unrelated earlier call's result (a launch checked with cudaGetLastError reported those).
template <typename... KArgs, typename... Args>
cudaError_t launch_plain(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Records e as the CUDA error behind the calling thread's latest GDR_ERR_CUDA (gdr_last_cuda_error) and
// returns GDR_ERR_CUDA.
gdr_status cuda_fail(cudaError_t e);

// Recurrent decode: T tokens of B sequences applied one by one to the fp32 states (state_in may be null
// for zero states and may alias state_out); o [B,T,Hv,V].
cudaError_t launch_decode(const Args &a, const void *q, const void *k, const void *v, const void *g,
                          const void *beta, const float *state_in, float *state_out, void *o, cudaStream_t s);

// Gate and beta activations (GDR_GATE_IN_KERNEL, GDR_BETA_SIGMOID_IN_KERNEL, GDR_ALLOW_NEG_EIGVAL) over the
// [tokens, Hv] scalars: the forward's activated g, beta (fp32) and sigmoid(-x) (sg, nullable); the backward's
// activated beta; and the backward's gradients w.r.t. the raw g and beta (in the gate dtype) from those w.r.t.
// the activated ones.  a.gate_f32 describes the raw tensors.
cudaError_t launch_gate_act_fwd(const Args &a, const void *g, const void *beta, unsigned flags, float *geff,
                                float *beff, float *sg, cudaStream_t s);
cudaError_t launch_gate_act_beta(const Args &a, const void *beta, unsigned flags, float *beff, cudaStream_t s);
cudaError_t launch_gate_act_bwd(const Args &a, const float *dgeff, const float *dbeff, const float *sg,
                                const void *beta, unsigned flags, void *dg, void *dbeta, cudaStream_t s);

// Zero padding of head dimensions below 128 (pad.cu): fp32 states [nh, R, Cc] <-> [nh, 128, 128] (Cc a
// multiple of 4).
cudaError_t launch_pad_state(const float *src, float *dst, long long nh, int R, int Cc, cudaStream_t s);
cudaError_t launch_unpad_state(const float *src, float *dst, long long nh, int R, int Cc, cudaStream_t s);

cudaError_t launch_prep_chunks(const int32_t *cu, int N, int T, int chunk, int32_t *idx, int64_t max_chunks,
                               int32_t *off, int32_t *total, int32_t *order, int bad_total, unsigned *err,
                               cudaStream_t s);

// Forward: per-chunk gate cumsum, WY matrix A and (P != nullptr) the decayed causal attention block
// P = scale (q^ k^T o Gamma) [tokens,Hv,64] with the inverse q/k norms rq, rk [tokens,Hv] (written only
// with in-kernel L2 normalisation).
cudaError_t launch_wy_fwd(const Args &a, const void *q, const void *k, const void *g, const void *beta, float *g_cs,
                          void *A, void *P, float *rq, float *rk, cudaStream_t s);
// The same P, rq, rk from a given g_cumsum (no A), on tcgen05 (one persistent CTA per SM).
cudaError_t launch_chunk_p_tc(const Args &a, const void *q, const void *k, const float *g_cs, void *P, float *rq,
                              float *rk, cudaStream_t s);
// Forward recurrence + output (o != nullptr) and/or per-chunk states (h != nullptr)
// and per-chunk Delta = U - W h (delta != nullptr).
cudaError_t launch_chain_fwd(const Args &a, const void *q, const void *k, const void *v, const float *g_cs,
                             const void *beta, const void *A, const float *h0, void *o, float *final_state, void *h,
                             bool h_api_layout, void *delta, const SegWs &sw, cudaStream_t s);
// Forward recurrence, warp-specialised (one CTA per value-column slice, and per segment of the intra-GPU
// split when nseg > 1).  o != nullptr: output rows; h: state before every chunk ([rows,Hv,K,V], or [..,V,K]
// when h_vfirst); delta: Delta of every chunk; seg_start: transposed fp32 start states [N,Hv,nseg,V,K]
// replacing h0 (from launch_chain_fwd_affine).  P, rq, rk: from launch_wy_fwd / launch_chunk_p_tc (P is read
// only when o != nullptr; rq, rk only with in-kernel L2 normalisation).
cudaError_t launch_chain_ws(const Args &a, const void *q, const void *k, const void *v, const float *g_cs,
                            const void *beta, const void *A, const void *P, const float *rq, const float *rk,
                            const float *h0, const float *seg_start, int nseg, void *o, float *final_state, void *h,
                            bool h_vfirst, void *delta, cudaStream_t s);
// The forward's segment-affine pass of the intra-GPU split on the warp-specialised chain (whole-width CTAs, no
// output; block x = kind): every segment's end state from a zero start (end0) and from the identity with
// zero values (end1), transposed [N,Hv,nseg,V,K] fp32.  rq, rk: with in-kernel L2 normalisation.
cudaError_t launch_chain_ws_affine(const Args &a, const void *q, const void *k, const void *v, const float *g_cs,
                                   const void *beta, const void *A, const float *rq, const float *rk, int nseg,
                                   float *end0, float *end1, cudaStream_t s);
// The forward segment scan alone (sw.end0, sw.end1 -> sw.start, from h0).
cudaError_t launch_fwd_compose(const Args &a, const float *h0, const SegWs &sw, cudaStream_t s);
// The intra-GPU split's first two steps (sw.nseg > 1): the segment-affine passes and the scan, leaving the
// start state of every segment in sw.start (forward: from h0; reverse: the gradient at every segment's end,
// from dht).
cudaError_t launch_chain_fwd_affine(const Args &a, const void *q, const void *k, const void *v, const float *g_cs,
                                    const void *beta, const void *A, const float *h0, const SegWs &sw, cudaStream_t s);
cudaError_t launch_chain_bwd_affine(const Args &a, const void *q, const void *k, const float *g_cs, const void *beta,
                                    const void *A, const void *dout, const float *dht, const SegWs &sw, cudaStream_t s);
// Backward without a sequence split, warp-specialised: the forward recompute (states h and Delta of every
// chunk, no output) and the reverse chain (dH' and dDelta of every chunk, dh0) in one launch, one CTA each
// per (sequence, value head).  P, rq, rk from launch_chunk_p_tc.
cudaError_t launch_chain_ws_pair(const Args &a, const void *q, const void *k, const void *v, const float *g_cs,
                                 const void *beta, const void *A, const void *P, const float *rq, const float *rk,
                                 const float *h0, void *h, void *delta, const void *dout, const float *dht,
                                 void *dhn, void *ddelta, float *dh0, cudaStream_t s);
// The reverse chain alone (dH' and dDelta of every chunk (each nullable), dh0), warp-specialised, one CTA per
// (sequence, value head, 64-column slice or whole width, and segment when nseg > 1); for callers that hold the
// forward's states and Delta.  seg_start: the gradients at the segments' ends [N,Hv,nseg,V,K] (from the
// scan), replacing dht.  seg_end (nullable): every segment's gradient at its start, [N,Hv,nseg,V,K], in
// place of dh0 (with dht and seg_start NULL: the split's zero-start reverse pass).  P, rq, rk as for
// launch_chain_ws_pair.
cudaError_t launch_chain_rev(const Args &a, const void *q, const void *k, const float *g_cs, const void *beta,
                             const void *A, const void *P, const float *rq, const float *rk, const void *dout,
                             const float *dht, const float *seg_start, int nseg, void *dhn, void *ddelta, float *dh0,
                             float *seg_end, cudaStream_t s);
// The reverse scan of the split from the segments' zero-start gradients (sw.end0) and the forward's transfer
// matrices fwd_transfer [N,Hv,nseg,V,K] (transposed into sw.end1): the gradient at every segment's end into
// sw.start.
cudaError_t launch_rev_compose(const Args &a, const float *dht, const float *fwd_transfer, const SegWs &sw,
                               cudaStream_t s);
// Backward: reverse state-gradient chain (dH' and dDelta of every chunk, dh0).
cudaError_t launch_chain_bwd(const Args &a, const void *q, const void *k, const float *g_cs, const void *beta,
                             const void *A, const void *dout, const float *dht, void *dhn, void *ddelta, float *dh0,
                             const SegWs &sw, cudaStream_t s);
// Backward, after launch_bwd_chunk_tc: for sequences of one chunk, the dg correction from the fp32 h0 and dht
// (onechunk.cu); dg in the gate dtype (a.gate_f32) or fp32.
cudaError_t launch_onechunk_dg(const Args &a, const float *h0, const float *dht, const float *g_cs, void *dg,
                               cudaStream_t s);
// Backward: per-chunk gradients (dq, dk, dv, dg, dbeta).
cudaError_t launch_bwd_chunk_tc(const Args &a, const void *q, const void *k, const void *v, const float *g_cs,
                                const void *beta, const void *A, const void *dout, const void *h, const void *dhn,
                                const void *delta, const void *ddelta, void *dq, void *dk, void *dv, void *dg,
                                void *dbeta, cudaStream_t s);

}  // namespace gdr
