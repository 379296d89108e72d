/*
 * Float64 CPU oracle for the gated delta rule (GDN and KDA), forward and
 * reverse mode.  TEST INFRASTRUCTURE ONLY: nothing on the CUDA product path
 * links, calls or includes this file; only the tests, the smoke check and the
 * benchmark's CPU-baseline leg use it.
 *
 * What it computes (plain definition, token by token, no chunking):
 *
 *   recurrence (the gated delta rule with the decay applied before the
 *   delta update -- the order the FlashKDA derived quantities kd = k*e^{gc},
 *   ki = k*e^{-gc}, kr = k*e^{gT-gc} imply; "FlashKDA之backward（K1）", §3.2 and
 *   the kernel's workspace comments; for a scalar gate both orders coincide):
 *
 *     qn = q / sqrt(|q|^2 + 1e-6),  kn = k / sqrt(|k|^2 + 1e-6)
 *                                  ("FlashKDA之backward（K1）", §3.1: L2 norm
 *                                   with eps 1e-6 inside the square root)
 *     beta = sigmoid(b)            (same page, §6: gradient returned in logit space)
 *     St  = diag(exp(g_t)) S_{t-1}                 (g_t: per-channel log gate)
 *     p   = St^T kn
 *     u   = beta * (v - p)
 *     S_t = St + kn u^T
 *     o_t = scale * S_t^T qn
 *
 *   The state S is D x D with rows indexed by the key channel and columns by
 *   the value channel.  The loss whose gradient is returned is
 *     L = sum_t <dO_t, o_t> + sum_seq <dht, S_T>.
 *
 *   Reverse mode, per token from last to first (hand derived from the lines
 *   above; each line is the adjoint of one forward line):
 *     dqn  = scale * S_t dO_t ;          dS += scale * qn dO_t^T
 *     dkn  = dS u ;                      du  = dS^T kn
 *     dbeta = <du, v - p> ;  dv = beta du ;  dp = -beta du
 *     dkn += St dp ;                     dSt = dS + kn dp^T
 *     dg_t[d] = sum_j dSt[d][j] * St[d][j]
 *     dS   = diag(exp(g_t)) dSt
 *   then dh0 = dS, the L2-norm backward (dx = (dxn - xn <dxn, xn>) / |x|,
 *   "FlashKDA之backward（K1）", §3.3) and dlogit = dbeta * beta * (1 - beta)
 *   (same page, §6).
 *
 * Gate input: glog is the per-channel natural-log gate [T,H,D].  The GDN
 * scalar gate is passed broadcast over the channels and its gradient is the
 * channel sum; the KDA gate function and its chain rule live in oracle.py.
 *
 * Memory: the state is checkpointed every BLK tokens during the forward pass
 * and the BLK states of one block are recomputed during the reverse pass.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define BLK 64

typedef struct {
    int H, D;
    double scale;
    const double *q, *k, *v, *glog, *blogit, *h0, *dO, *dht;
    double *o, *ht, *dq, *dk, *dv, *dglog, *dblogit, *dh0;
} job_t;

static double l2_inv(const double* x, int D) {
    double s = 0.0;
    for (int i = 0; i < D; ++i) s += x[i] * x[i];
    return 1.0 / sqrt(s + 1e-6);
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* One token of the forward recurrence.  S_prev -> S_next; also returns the
 * decayed state St, p, u and beta (the quantities the reverse step needs). */
static void fwd_token(const job_t* J, int64_t t, int h, const double* S_prev, double* St,
                      double* S_next, double* p, double* u, double* kn, double* qn,
                      double* beta_out) {
    const int D = J->D, H = J->H;
    const int64_t base = (t * H + h) * (int64_t)D;
    const double* kt = J->k + base;
    const double* qt = J->q + base;
    const double* vt = J->v + base;
    const double* gt = J->glog + base;
    double ik = l2_inv(kt, D), iq = l2_inv(qt, D);
    for (int d = 0; d < D; ++d) { kn[d] = kt[d] * ik; qn[d] = qt[d] * iq; }
    double beta = sigmoid(J->blogit[t * H + h]);
    for (int j = 0; j < D; ++j) p[j] = 0.0;
    for (int d = 0; d < D; ++d) {
        double a = exp(gt[d]);
        const double* sr = S_prev + (int64_t)d * D;
        double* tr = St + (int64_t)d * D;
        for (int j = 0; j < D; ++j) { tr[j] = a * sr[j]; p[j] += tr[j] * kn[d]; }
    }
    for (int j = 0; j < D; ++j) u[j] = beta * (vt[j] - p[j]);
    for (int d = 0; d < D; ++d) {
        const double* tr = St + (int64_t)d * D;
        double* nr = S_next + (int64_t)d * D;
        for (int j = 0; j < D; ++j) nr[j] = tr[j] + kn[d] * u[j];
    }
    *beta_out = beta;
}

static void run_pair(const job_t* J, int64_t bos, int64_t len, int seq, int h) {
    const int D = J->D, H = J->H;
    const int64_t DD = (int64_t)D * D;
    const int want_bwd = (J->dO != NULL);
    const int64_t nblk = (len + BLK - 1) / BLK;

    double* ckpt = (double*)calloc((size_t)(nblk + 1) * DD, sizeof(double));
    double* S = (double*)malloc(sizeof(double) * DD);
    double* St = (double*)malloc(sizeof(double) * DD);
    double* Sn = (double*)malloc(sizeof(double) * DD);
    double* vec = (double*)malloc(sizeof(double) * 16 * D);
    double *p = vec, *u = vec + D, *kn = vec + 2 * D, *qn = vec + 3 * D;
    double *dqn = vec + 4 * D, *dkn = vec + 5 * D, *du = vec + 6 * D, *dp = vec + 7 * D;

    const int64_t sbase = ((int64_t)seq * H + h) * DD;
    if (J->h0) memcpy(S, J->h0 + sbase, sizeof(double) * DD);
    else memset(S, 0, sizeof(double) * DD);

    /* forward: outputs and checkpoints */
    for (int64_t i = 0; i < len; ++i) {
        if (i % BLK == 0) memcpy(ckpt + (i / BLK) * DD, S, sizeof(double) * DD);
        double beta;
        int64_t t = bos + i;
        fwd_token(J, t, h, S, St, Sn, p, u, kn, qn, &beta);
        if (J->o) {
            double* ot = J->o + (t * H + h) * (int64_t)D;
            for (int j = 0; j < D; ++j) ot[j] = 0.0;
            for (int d = 0; d < D; ++d) {
                const double* nr = Sn + (int64_t)d * D;
                for (int j = 0; j < D; ++j) ot[j] += nr[j] * qn[d];
            }
            for (int j = 0; j < D; ++j) ot[j] *= J->scale;
        }
        double* tmp = S; S = Sn; Sn = tmp;
    }
    if (J->ht) memcpy(J->ht + sbase, S, sizeof(double) * DD);

    if (want_bwd) {
        double* dS = (double*)malloc(sizeof(double) * DD);
        double* blk = (double*)malloc(sizeof(double) * (BLK + 1) * DD);
        if (J->dht) memcpy(dS, J->dht + sbase, sizeof(double) * DD);
        else memset(dS, 0, sizeof(double) * DD);

        for (int64_t b = nblk - 1; b >= 0; --b) {
            int64_t i0 = b * BLK, i1 = i0 + BLK < len ? i0 + BLK : len;
            /* recompute the states S_{i0-1} .. S_{i1-1} of this block */
            memcpy(blk, ckpt + b * DD, sizeof(double) * DD);
            for (int64_t i = i0; i < i1; ++i) {
                double beta;
                fwd_token(J, bos + i, h, blk + (i - i0) * DD, St, blk + (i - i0 + 1) * DD, p, u,
                          kn, qn, &beta);
            }
            for (int64_t i = i1 - 1; i >= i0; --i) {
                const int64_t t = bos + i;
                const int64_t base = (t * H + h) * (int64_t)D;
                const double* Sprev = blk + (i - i0) * DD;
                const double* Snew = blk + (i - i0 + 1) * DD;
                double beta;
                fwd_token(J, t, h, Sprev, St, Sn, p, u, kn, qn, &beta);
                const double* dOt = J->dO + base;
                const double* gt = J->glog + base;
                const double* vt = J->v + base;
                /* o = scale * S_t^T qn */
                for (int d = 0; d < D; ++d) {
                    const double* nr = Snew + (int64_t)d * D;
                    double acc = 0.0;
                    for (int j = 0; j < D; ++j) acc += nr[j] * dOt[j];
                    dqn[d] = J->scale * acc;
                    double* g = dS + (int64_t)d * D;
                    double c = J->scale * qn[d];
                    for (int j = 0; j < D; ++j) g[j] += c * dOt[j];
                }
                /* S_t = St + kn u^T */
                for (int j = 0; j < D; ++j) du[j] = 0.0;
                for (int d = 0; d < D; ++d) {
                    const double* g = dS + (int64_t)d * D;
                    double acc = 0.0;
                    for (int j = 0; j < D; ++j) { acc += g[j] * u[j]; du[j] += g[j] * kn[d]; }
                    dkn[d] = acc;
                }
                /* u = beta (v - p) */
                double dbeta = 0.0;
                for (int j = 0; j < D; ++j) {
                    dbeta += du[j] * (vt[j] - p[j]);
                    J->dv[base + j] = beta * du[j];
                    dp[j] = -beta * du[j];
                }
                /* p = St^T kn ; St = diag(exp g) S_prev */
                for (int d = 0; d < D; ++d) {
                    const double* tr = St + (int64_t)d * D;
                    double* g = dS + (int64_t)d * D;
                    double a = exp(gt[d]);
                    double acc = 0.0, dgd = 0.0;
                    for (int j = 0; j < D; ++j) {
                        acc += tr[j] * dp[j];
                        double dst = g[j] + kn[d] * dp[j];
                        dgd += dst * tr[j];
                        g[j] = a * dst;
                    }
                    dkn[d] += acc;
                    J->dglog[base + d] = dgd;
                }
                /* L2-norm backward and the sigmoid of beta */
                const double* qt = J->q + base;
                const double* kt = J->k + base;
                double iq = l2_inv(qt, D), ik = l2_inv(kt, D);
                double sq = 0.0, sk = 0.0;
                for (int d = 0; d < D; ++d) { sq += dqn[d] * qn[d]; sk += dkn[d] * kn[d]; }
                for (int d = 0; d < D; ++d) {
                    J->dq[base + d] = (dqn[d] - qn[d] * sq) * iq;
                    J->dk[base + d] = (dkn[d] - kn[d] * sk) * ik;
                }
                J->dblogit[t * H + h] = dbeta * beta * (1.0 - beta);
            }
        }
        memcpy(J->dh0 + sbase, dS, sizeof(double) * DD);
        free(blk);
        free(dS);
    }
    free(vec); free(Sn); free(St); free(S); free(ckpt);
}

/*
 * Runs every (sequence, head) pair.  cu_seqlens: host int64 [N+1] offsets into
 * the token axis.  All tensors are host float64, token-major:
 *   q, k, v, glog, dO, o, dq, dk, dv, dglog : [T_total, H, D]
 *   blogit, dblogit                         : [T_total, H]
 *   h0, dht, ht, dh0                        : [N, H, D, D]  (row = key channel)
 * h0 / dht may be NULL (zero).  dO == NULL runs the forward only; otherwise
 * dq, dk, dv, dglog, dblogit, dh0 must all be non-NULL.  o / ht may be NULL.
 * nthreads <= 0 uses the OpenMP default.  Returns 0, or -1 on bad arguments.
 */
int oracle_gdr(int N, const int64_t* cu_seqlens, int H, int D, double scale, const double* q,
               const double* k, const double* v, const double* glog, const double* blogit,
               const double* h0, const double* dO, const double* dht, double* o, double* ht,
               double* dq, double* dk, double* dv, double* dglog, double* dblogit, double* dh0,
               int nthreads) {
    if (N < 0 || H <= 0 || D <= 0 || !cu_seqlens || !q || !k || !v || !glog || !blogit) return -1;
    if (dO && (!dq || !dk || !dv || !dglog || !dblogit || !dh0)) return -1;
    for (int s = 0; s < N; ++s)
        if (cu_seqlens[s + 1] < cu_seqlens[s]) return -1;
    job_t J = {H, D, scale, q, k, v, glog, blogit, h0, dO, dht, o, ht, dq, dk, dv, dglog, dblogit, dh0};
    const int64_t npairs = (int64_t)N * H;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t pi = 0; pi < npairs; ++pi) {
        int seq = (int)(pi / H), h = (int)(pi % H);
        run_pair(&J, cu_seqlens[seq], cu_seqlens[seq + 1] - cu_seqlens[seq], seq, h);
    }
    return 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
