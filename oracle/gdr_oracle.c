/*
 * Oracle for the chunked Gated Delta Rule -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark may load this file's library.  The product path (the CUDA
 * library) never calls it and shares no code with it.
 *
 * What it computes: the gated delta rule, one token at a time, in fp64.
 * The state is kept in the [K,V] layout of the state tensors:
 *
 *     h_t = exp(g_t) (I - beta_t k_t k_t^T) h_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * h_t^T q_t
 *
 * This is the transposed form of the recurrence stated for the method
 * ("Gated Delta Rule" op, FlashQLA skill page, "Core API" section: q,k
 * [B,T,H_q,K], v [B,T,H_v,V], g "gate (exponential decay)", beta "delta
 * rule beta coefficient", state [B,H_v,K,V]).  It is evaluated in the
 * equivalent "delta" form
 *
 *     p = k^T h_{t-1};  delta = beta (v - e^g p);  h_t = e^g h_{t-1} + k delta^T
 *
 * The backward pass is plain reverse-mode differentiation of that token
 * loop, with the state checkpointed at every chunk boundary and the states
 * of one chunk recomputed from its checkpoint.
 *
 * Options follow the op's keyword arguments (PR #998 "[GDN] Add FlashQLA
 * backend dispatch", Summary and review threads): optional per-token L2
 * normalisation of q and k ("use_qk_l2norm_in_kernel"; x / sqrt(sum x^2 + eps)
 * with eps = 1e-6, a reading: the pages do not give eps), state_v_first
 * (every state-shaped tensor stored [V,K] instead of [K,V]), variable-length
 * packed batches, and grouped value attention (v-head j reads q/k head
 * j / (H_v/H_q)).
 *
 * Layout: tokens are packed; sequence n owns tokens [start[n], start[n]+len[n]).
 * q,k: [Ttot,Hq,K]; v,o: [Ttot,Hv,V]; g,beta: [Ttot,Hv];
 * states: [N,Hv,K,V] (or [N,Hv,V,K] with state_v_first).
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef long long i64;

#define L2_EPS 1e-6

/* x -> x / sqrt(sum x^2 + eps) when on, else copy.  Returns the norm used. */
static double normalise(const double *x, int D, int on, double *out) {
    if (!on) {
        memcpy(out, x, sizeof(double) * (size_t)D);
        return 1.0;
    }
    double ss = 0.0;
    for (int d = 0; d < D; ++d) ss += x[d] * x[d];
    double n = sqrt(ss + L2_EPS);
    for (int d = 0; d < D; ++d) out[d] = x[d] / n;
    return n;
}

/* Read a state block [K,V] (or stored [V,K] when vf) into h[K][V]. */
static void load_state(const double *src, int K, int V, int vf, double *h) {
    if (!vf) {
        memcpy(h, src, sizeof(double) * (size_t)K * V);
    } else {
        for (int d = 0; d < K; ++d)
            for (int e = 0; e < V; ++e) h[(size_t)d * V + e] = src[(size_t)e * K + d];
    }
}

static void store_state(double *dst, int K, int V, int vf, const double *h) {
    if (!vf) {
        memcpy(dst, h, sizeof(double) * (size_t)K * V);
    } else {
        for (int d = 0; d < K; ++d)
            for (int e = 0; e < V; ++e) dst[(size_t)e * K + d] = h[(size_t)d * V + e];
    }
}

/* One token of the recurrence.  h is updated in place; p, delta returned. */
static void step(double *h, const double *kh, const double *vt, double a, double b, int K, int V,
                 double *p, double *delta) {
    for (int e = 0; e < V; ++e) p[e] = 0.0;
    for (int d = 0; d < K; ++d) {
        const double kd = kh[d];
        const double *hd = h + (size_t)d * V;
        for (int e = 0; e < V; ++e) p[e] += kd * hd[e];
    }
    for (int e = 0; e < V; ++e) delta[e] = b * (vt[e] - a * p[e]);
    for (int d = 0; d < K; ++d) {
        const double kd = kh[d];
        double *hd = h + (size_t)d * V;
        for (int e = 0; e < V; ++e) hd[e] = a * hd[e] + kd * delta[e];
    }
}

/*
 * Forward.  head_sel (nullable) picks the v-heads to evaluate; outputs of the
 * other heads are left untouched.  h_chunks (nullable) receives the state
 * before every chunk of `chunk` tokens: row chunk_base[n] + c for chunk c of
 * sequence n, layout [rows,Hv,K,V] (or [.., V,K] with vf).  delta_out
 * (nullable) receives the per-token delta [Ttot,Hv,V].
 */
int gdr_oracle_fwd(int N, const i64 *seq_start, const i64 *seq_len, int Hq, int Hv, int K, int V,
                   double scale, int l2norm, int vf, int chunk, const double *q, const double *k,
                   const double *v, const double *g, const double *beta, const double *h0,
                   const unsigned char *head_sel, double *o, double *ht, double *h_chunks,
                   const i64 *chunk_base, double *delta_out, int nthreads) {
    if (N < 0 || Hq <= 0 || Hv <= 0 || K <= 0 || V <= 0 || Hv % Hq != 0 || chunk <= 0) return 1;
    const int grp = Hv / Hq;
    const i64 npairs = (i64)N * Hv;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
    int err = 0;
#pragma omp parallel
    {
        double *h = (double *)malloc(sizeof(double) * (size_t)K * V);
        double *qh = (double *)malloc(sizeof(double) * (size_t)K);
        double *kh = (double *)malloc(sizeof(double) * (size_t)K);
        double *p = (double *)malloc(sizeof(double) * (size_t)V);
        double *dl = (double *)malloc(sizeof(double) * (size_t)V);
        if (!h || !qh || !kh || !p || !dl) {
#pragma omp atomic write
            err = 2;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (i64 pr = 0; pr < npairs; ++pr) {
                const int n = (int)(pr / Hv), j = (int)(pr % Hv), i = j / grp;
                if (head_sel && !head_sel[j]) continue;
                const i64 s0 = seq_start[n], L = seq_len[n];
                if (h0)
                    load_state(h0 + ((size_t)n * Hv + j) * K * V, K, V, vf, h);
                else
                    memset(h, 0, sizeof(double) * (size_t)K * V);
                for (i64 u = 0; u < L; ++u) {
                    const i64 t = s0 + u;
                    if (h_chunks && u % chunk == 0)
                        store_state(h_chunks + ((size_t)(chunk_base[n] + u / chunk) * Hv + j) * K * V,
                                    K, V, vf, h);
                    normalise(q + ((size_t)t * Hq + i) * K, K, l2norm, qh);
                    normalise(k + ((size_t)t * Hq + i) * K, K, l2norm, kh);
                    const double a = exp(g[(size_t)t * Hv + j]);
                    const double b = beta[(size_t)t * Hv + j];
                    step(h, kh, v + ((size_t)t * Hv + j) * V, a, b, K, V, p, dl);
                    double *ot = o + ((size_t)t * Hv + j) * V;
                    for (int e = 0; e < V; ++e) ot[e] = 0.0;
                    for (int d = 0; d < K; ++d) {
                        const double qd = qh[d];
                        const double *hd = h + (size_t)d * V;
                        for (int e = 0; e < V; ++e) ot[e] += hd[e] * qd;
                    }
                    for (int e = 0; e < V; ++e) ot[e] *= scale;
                    if (delta_out) memcpy(delta_out + ((size_t)t * Hv + j) * V, dl, sizeof(double) * V);
                }
                if (ht) store_state(ht + ((size_t)n * Hv + j) * K * V, K, V, vf, h);
            }
        }
        free(h); free(qh); free(kh); free(p); free(dl);
    }
    return err;
}

/*
 * Backward: reverse-mode over the token loop of gdr_oracle_fwd.
 * dout [Ttot,Hv,V]; dht (nullable) the gradient of the final state.
 * Writes dq, dk [Ttot,Hq,K] (summed over the v-heads of each q/k head that
 * head_sel keeps), dv [Ttot,Hv,V], dg, dbeta [Ttot,Hv], dh0 (nullable) [N,Hv,K,V].
 * Parallel over (sequence, q/k head); the v-heads of a group are visited in
 * increasing order, so the group sums have a fixed order.
 */
int gdr_oracle_bwd(int N, const i64 *seq_start, const i64 *seq_len, int Hq, int Hv, int K, int V,
                   double scale, int l2norm, int vf, int chunk, const double *q, const double *k,
                   const double *v, const double *g, const double *beta, const double *h0,
                   const double *dout, const double *dht, const unsigned char *head_sel,
                   double *dq, double *dk, double *dv, double *dg, double *dbeta, double *dh0,
                   int nthreads) {
    if (N < 0 || Hq <= 0 || Hv <= 0 || K <= 0 || V <= 0 || Hv % Hq != 0 || chunk <= 0) return 1;
    const int grp = Hv / Hq;
    const i64 ngroups = (i64)N * Hq;
    const size_t KV = (size_t)K * V;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
    int err = 0;
#pragma omp parallel
    {
        double *dH = (double *)malloc(sizeof(double) * KV);
        double *blk = (double *)malloc(sizeof(double) * KV * (size_t)(chunk + 1));
        double *qh = (double *)malloc(sizeof(double) * (size_t)K);
        double *kh = (double *)malloc(sizeof(double) * (size_t)K);
        double *p = (double *)malloc(sizeof(double) * (size_t)V);
        double *dl = (double *)malloc(sizeof(double) * (size_t)V);
        double *ddl = (double *)malloc(sizeof(double) * (size_t)V);
        double *dp = (double *)malloc(sizeof(double) * (size_t)V);
        double *ps = (double *)malloc(sizeof(double) * (size_t)V * chunk);
        double *dls = (double *)malloc(sizeof(double) * (size_t)V * chunk);
        if (!dH || !blk || !qh || !kh || !p || !dl || !ddl || !dp || !ps || !dls) {
#pragma omp atomic write
            err = 2;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (i64 gi = 0; gi < ngroups; ++gi) {
                const int n = (int)(gi / Hq), i = (int)(gi % Hq);
                const i64 s0 = seq_start[n], L = seq_len[n];
                /* gradients w.r.t. the normalised q/k of this group */
                double *dqh = (double *)calloc((size_t)(L > 0 ? L : 1) * K, sizeof(double));
                double *dkh = (double *)calloc((size_t)(L > 0 ? L : 1) * K, sizeof(double));
                const i64 nck = (L + chunk - 1) / chunk;
                double *ck = (double *)malloc(sizeof(double) * KV * (size_t)(nck > 0 ? nck : 1));
                if (!dqh || !dkh || !ck) {
#pragma omp atomic write
                    err = 2;
                    free(dqh); free(dkh); free(ck);
                    continue;
                }
                int any = 0;
                for (int jj = 0; jj < grp; ++jj) {
                    const int j = i * grp + jj;
                    if (head_sel && !head_sel[j]) continue;
                    any = 1;
                    /* forward, keeping the state before each chunk */
                    if (h0)
                        load_state(h0 + ((size_t)n * Hv + j) * KV, K, V, vf, blk);
                    else
                        memset(blk, 0, sizeof(double) * KV);
                    for (i64 u = 0; u < L; ++u) {
                        const i64 t = s0 + u;
                        if (u % chunk == 0) memcpy(ck + (size_t)(u / chunk) * KV, blk, sizeof(double) * KV);
                        normalise(k + ((size_t)t * Hq + i) * K, K, l2norm, kh);
                        step(blk, kh, v + ((size_t)t * Hv + j) * V, exp(g[(size_t)t * Hv + j]),
                             beta[(size_t)t * Hv + j], K, V, p, dl);
                    }
                    if (dht)
                        load_state(dht + ((size_t)n * Hv + j) * KV, K, V, vf, dH);
                    else
                        memset(dH, 0, sizeof(double) * KV);
                    for (i64 c = nck - 1; c >= 0; --c) {
                        const i64 u0 = c * chunk;
                        const int bl = (int)((L - u0) < chunk ? (L - u0) : chunk);
                        /* recompute the states of this chunk: blk[u] = state before token u0+u */
                        memcpy(blk, ck + (size_t)c * KV, sizeof(double) * KV);
                        for (int u = 0; u < bl; ++u) {
                            const i64 t = s0 + u0 + u;
                            memcpy(blk + (size_t)(u + 1) * KV, blk + (size_t)u * KV, sizeof(double) * KV);
                            normalise(k + ((size_t)t * Hq + i) * K, K, l2norm, kh);
                            step(blk + (size_t)(u + 1) * KV, kh, v + ((size_t)t * Hv + j) * V,
                                 exp(g[(size_t)t * Hv + j]), beta[(size_t)t * Hv + j], K, V,
                                 ps + (size_t)u * V, dls + (size_t)u * V);
                        }
                        for (int u = bl - 1; u >= 0; --u) {
                            const i64 t = s0 + u0 + u;
                            const double *hprev = blk + (size_t)u * KV;
                            const double *hcur = blk + (size_t)(u + 1) * KV;
                            const double *pt = ps + (size_t)u * V;
                            const double *dlt = dls + (size_t)u * V;
                            const double *dot = dout + ((size_t)t * Hv + j) * V;
                            const double *vt = v + ((size_t)t * Hv + j) * V;
                            const double a = exp(g[(size_t)t * Hv + j]);
                            const double b = beta[(size_t)t * Hv + j];
                            normalise(q + ((size_t)t * Hq + i) * K, K, l2norm, qh);
                            normalise(k + ((size_t)t * Hq + i) * K, K, l2norm, kh);
                            double *dqt = dqh + (size_t)(u0 + u) * K;
                            double *dkt = dkh + (size_t)(u0 + u) * K;
                            /* o_t = scale h_t^T q */
                            for (int d = 0; d < K; ++d) {
                                double s = 0.0;
                                const double *hd = hcur + (size_t)d * V;
                                for (int e = 0; e < V; ++e) s += hd[e] * dot[e];
                                dqt[d] += scale * s;
                            }
                            for (int d = 0; d < K; ++d) {
                                double *dHd = dH + (size_t)d * V;
                                const double sq = scale * qh[d];
                                for (int e = 0; e < V; ++e) dHd[e] += sq * dot[e];
                            }
                            /* h_t = a h_{t-1} + k delta^T */
                            for (int e = 0; e < V; ++e) ddl[e] = 0.0;
                            double da = 0.0;
                            for (int d = 0; d < K; ++d) {
                                const double *dHd = dH + (size_t)d * V;
                                const double *hp = hprev + (size_t)d * V;
                                double s = 0.0;
                                for (int e = 0; e < V; ++e) {
                                    s += dHd[e] * dlt[e];
                                    ddl[e] += dHd[e] * kh[d];
                                    da += dHd[e] * hp[e];
                                }
                                dkt[d] += s;
                            }
                            /* delta = b (v - a p) */
                            double db = 0.0;
                            double *dvt = dv + ((size_t)t * Hv + j) * V;
                            for (int e = 0; e < V; ++e) {
                                db += ddl[e] * (vt[e] - a * pt[e]);
                                dvt[e] = b * ddl[e];
                                da -= b * ddl[e] * pt[e];
                                dp[e] = -b * a * ddl[e];
                            }
                            /* p = k^T h_{t-1} */
                            for (int d = 0; d < K; ++d) {
                                const double *hp = hprev + (size_t)d * V;
                                double s = 0.0;
                                for (int e = 0; e < V; ++e) s += hp[e] * dp[e];
                                dkt[d] += s;
                            }
                            for (int d = 0; d < K; ++d) {
                                double *dHd = dH + (size_t)d * V;
                                for (int e = 0; e < V; ++e) dHd[e] = a * dHd[e] + kh[d] * dp[e];
                            }
                            dbeta[(size_t)t * Hv + j] = db;
                            dg[(size_t)t * Hv + j] = a * da;
                        }
                    }
                    if (dh0) store_state(dh0 + ((size_t)n * Hv + j) * KV, K, V, vf, dH);
                }
                if (any) {
                    /* chain rule through x / sqrt(sum x^2 + eps) */
                    for (i64 u = 0; u < L; ++u) {
                        const i64 t = s0 + u;
                        for (int w = 0; w < 2; ++w) {
                            const double *x = (w == 0 ? q : k) + ((size_t)t * Hq + i) * K;
                            const double *dxh = (w == 0 ? dqh : dkh) + (size_t)u * K;
                            double *dx = (w == 0 ? dq : dk) + ((size_t)t * Hq + i) * K;
                            if (!l2norm) {
                                memcpy(dx, dxh, sizeof(double) * K);
                                continue;
                            }
                            double *xh = (w == 0 ? qh : kh);
                            const double nrm = normalise(x, K, 1, xh);
                            double dot = 0.0;
                            for (int d = 0; d < K; ++d) dot += xh[d] * dxh[d];
                            for (int d = 0; d < K; ++d) dx[d] = (dxh[d] - xh[d] * dot) / nrm;
                        }
                    }
                }
                free(dqh); free(dkh); free(ck);
            }
        }
        free(dH); free(blk); free(qh); free(kh); free(p); free(dl); free(ddl); free(dp); free(ps); free(dls);
    }
    return err;
}

int gdr_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
