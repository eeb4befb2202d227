/*
 * gdn_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU restatement of the Gated DeltaNet forward and of its
 * span summary, written token by token from the definitions on the cuDNN
 * "Linear Attention" operations page (sections "Layout", "Semantics worth
 * knowing": States and checkpoints, Summaries).  It is the parity oracle for
 * the CUDA path and shares no code with it.  Only tests/, the smoke check and
 * the CPU-baseline leg of bench.py may load it; the library never does.
 *
 * Per (sequence i, output head h), with tokens t = cu[i] .. cu[i+1]-1:
 *
 *     S_t = exp(g_t) * (I - beta_t k_t k_t^T) * S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * evaluated in the algebraically identical rank-1 order
 *     S <- exp(g) S ;  x = S^T k ;  S <- S + beta k (v - x)^T ;  o = scale S^T q
 * with q, k optionally L2-normalised first (x / sqrt(sum x^2 + 1e-6)) and the
 * scale applied after the normalisation.
 *
 * Grouped value heads: HO = HV output heads, q/k head = h / (HV / HK).
 * Checkpoints: the state *before* token offset j*n for j = 0 .. ceil(L/n)-1,
 * packed in sequence order (row = ckpt_off[i] + j).
 * Summary transition: P = prod_{t = L-1 .. 0} exp(g_t)(I - beta_t k_t k_t^T),
 * stored transposed (transition[i,h,a,b] = P[b][a]) so that
 *     S_final[b][v] = sum_a transition[a][b] * S_init[a][v] + S_H[b][v].
 *
 * Parity pins: every function here is pinned by tests/test_oracle_pins.py
 * against brute-force dense products, closed forms (retrieval, pure decay,
 * single token), linearity, span composition and hand-derived golden values;
 * the backward (gdn_oracle_bwd, at the end) against central finite differences
 * of the forward.
 *
 * `mutation` != 0 plants a deliberate mistake (a dropped term, a flipped sign,
 * a wrong index); it exists only so the pin tests can show that each planted
 * mistake is caught.  0 is the correct oracle.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    /* inputs, fp64, contiguous */
    const double *q;     /* [T, HK, K] */
    const double *k;     /* [T, HK, K] */
    const double *v;     /* [T, HV, V] */
    const double *g;     /* [T, HO]  natural-log decay */
    const double *beta;  /* [T, HO] */
    const int64_t *cu;   /* [N + 1] */
    int64_t T;
    int N, HK, HV, K, V;
    double scale;
    int l2norm;
    const double *s0;    /* [N, HO, K, V] or NULL (zero start) */
    /* outputs, fp64, contiguous, any may be NULL */
    double *o;           /* [T, HO, V] */
    double *final_state; /* [N, HO, K, V] */
    double *ckpt;        /* [R, HO, K, V] */
    int64_t ckpt_n;
    const int64_t *ckpt_off; /* [N] first checkpoint row of each sequence */
    double *transition;  /* [N, HO, K, K] */
    const unsigned char *unit_mask; /* [N * HO] or NULL: compute only marked units */
    int mutation;
    /* work distribution */
    int64_t next_unit;
    pthread_mutex_t lock;
} oracle_job;

static void l2_normalise(double *x, int n, int mutation) {
    double ss = 0.0;
    for (int d = 0; d < n; ++d) ss += x[d] * x[d];
    double r = 1.0 / sqrt(ss + 1e-6);
    if (mutation == 5) r = 1.0 / (ss + 1e-6); /* planted: missing sqrt */
    for (int d = 0; d < n; ++d) x[d] *= r;
}

static void run_unit(const oracle_job *J, int i, int h) {
    const int K = J->K, V = J->V, HO = J->HV, HK = J->HK;
    const int group = J->HV / J->HK;
    int hk = h / group;
    if (J->mutation == 6) hk = h % HK; /* planted: interleaved instead of contiguous GVA groups */
    const int64_t t0 = J->cu[i], t1 = J->cu[i + 1];
    const int64_t unit = (int64_t)i * HO + h;

    double *S = calloc((size_t)K * V, sizeof(double));
    double *P = J->transition ? calloc((size_t)K * K, sizeof(double)) : NULL;
    double *x = malloc(sizeof(double) * (size_t)(V > K ? V : K));
    double *qn = malloc(sizeof(double) * K);
    double *kn = malloc(sizeof(double) * K);
    if (J->s0) memcpy(S, J->s0 + unit * K * V, sizeof(double) * (size_t)K * V);
    if (P) for (int a = 0; a < K; ++a) P[a * K + a] = 1.0;

    for (int64_t t = t0; t < t1; ++t) {
        const int64_t off = t - t0;
        /* checkpoint entry j holds the state entering token offset j*n */
        int64_t ck_off = off;
        if (J->mutation == 8) ck_off = off - 1; /* planted: entries taken one token late */
        if (J->ckpt && ck_off >= 0 && ck_off % J->ckpt_n == 0) {
            const int64_t row = J->ckpt_off[i] + ck_off / J->ckpt_n;
            memcpy(J->ckpt + (row * HO + h) * K * V, S, sizeof(double) * (size_t)K * V);
        }
        memcpy(qn, J->q + (t * HK + hk) * K, sizeof(double) * K);
        memcpy(kn, J->k + (t * HK + hk) * K, sizeof(double) * K);
        if (J->l2norm) {
            l2_normalise(qn, K, J->mutation);
            l2_normalise(kn, K, J->mutation);
        }
        const double a = exp(J->g[t * HO + h]);
        const double b = J->beta[t * HO + h];
        const double *vt = J->v + (t * J->HV + h) * V;

        if (J->o && J->mutation == 4) { /* planted: exclusive output, reads S_{t-1} */
            double *ot = J->o + (t * HO + h) * V;
            for (int c = 0; c < V; ++c) {
                double acc = 0.0;
                for (int r = 0; r < K; ++r) acc += S[r * V + c] * qn[r];
                ot[c] = J->scale * acc;
            }
        }
        /* S <- exp(g) S */
        if (J->mutation != 1)
            for (int e = 0; e < K * V; ++e) S[e] *= a;
        /* x = S^T k */
        for (int c = 0; c < V; ++c) x[c] = 0.0;
        for (int r = 0; r < K; ++r)
            for (int c = 0; c < V; ++c) x[c] += S[r * V + c] * kn[r];
        /* S <- S + beta k (v - x)^T */
        for (int r = 0; r < K; ++r) {
            const double bk = b * kn[r];
            for (int c = 0; c < V; ++c) {
                double d = vt[c] - x[c];
                if (J->mutation == 2) d = vt[c] + x[c];  /* planted: erase sign flipped */
                if (J->mutation == 3) d = vt[c];         /* planted: erase term dropped */
                S[r * V + c] += bk * d;
            }
        }
        /* o = scale S^T q (inclusive: reads the state after token t) */
        if (J->o && J->mutation != 4) {
            double *ot = J->o + (t * HO + h) * V;
            for (int c = 0; c < V; ++c) {
                double acc = 0.0;
                for (int r = 0; r < K; ++r) acc += S[r * V + c] * qn[r];
                ot[c] = J->scale * acc;
            }
        }
        /* P <- exp(g) (I - beta k k^T) P */
        if (P) {
            for (int c = 0; c < K; ++c) {
                double y = 0.0;
                for (int r = 0; r < K; ++r) y += kn[r] * P[r * K + c];
                x[c] = y;
            }
            for (int r = 0; r < K; ++r)
                for (int c = 0; c < K; ++c)
                    P[r * K + c] = a * (P[r * K + c] - b * kn[r] * x[c]);
        }
    }
    if (J->final_state) memcpy(J->final_state + unit * K * V, S, sizeof(double) * (size_t)K * V);
    if (P) {
        double *Tr = J->transition + unit * K * K;
        for (int r = 0; r < K; ++r)
            for (int c = 0; c < K; ++c)
                Tr[c * K + r] = (J->mutation == 7) ? P[c * K + r] : P[r * K + c];
    }
    free(S); free(P); free(x); free(qn); free(kn);
}

static void *worker(void *arg) {
    oracle_job *J = (oracle_job *)arg;
    const int64_t units = (int64_t)J->N * J->HV;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int64_t u = J->next_unit++;
        pthread_mutex_unlock(&J->lock);
        if (u >= units) break;
        if (J->unit_mask && !J->unit_mask[u]) continue;
        run_unit(J, (int)(u / J->HV), (int)(u % J->HV));
    }
    return NULL;
}

/*
 * Entry point.  Returns 0 on success, -1 on an argument error.
 * All arrays are fp64 and contiguous; see oracle_job for shapes.
 */
int gdn_oracle_run(const double *q, const double *k, const double *v,
                   const double *g, const double *beta, const int64_t *cu,
                   int64_t T, int N, int HK, int HV, int K, int V,
                   double scale, int l2norm, const double *s0,
                   double *o, double *final_state,
                   double *ckpt, int64_t ckpt_n, const int64_t *ckpt_off,
                   double *transition, const unsigned char *unit_mask,
                   int nthreads, int mutation) {
    if (N < 0 || HK <= 0 || HV <= 0 || HV % HK != 0 || K <= 0 || V <= 0) return -1;
    if (cu[0] != 0 || cu[N] != T) return -1;
    for (int i = 0; i < N; ++i)
        if (cu[i + 1] < cu[i]) return -1;
    if (ckpt && (ckpt_n <= 0 || !ckpt_off)) return -1;

    oracle_job J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.cu = cu;
    J.T = T; J.N = N; J.HK = HK; J.HV = HV; J.K = K; J.V = V;
    J.scale = scale; J.l2norm = l2norm; J.s0 = s0;
    J.o = o; J.final_state = final_state;
    J.ckpt = ckpt; J.ckpt_n = ckpt_n; J.ckpt_off = ckpt_off;
    J.transition = transition; J.unit_mask = unit_mask;
    J.mutation = mutation;
    J.next_unit = 0;
    pthread_mutex_init(&J.lock, NULL);

    if (nthreads < 1) nthreads = 1;
    pthread_t *th = malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, worker, &J);
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    return 0;
}

/* ------------------------------------------------------------------------------------------
 * Backward (reverse mode) of the forward above, token by token in fp64.
 *
 * Inputs as for gdn_oracle_run plus do_ [T, HO, V] (dL/do) and dfinal [N, HO, K, V] (dL/dS
 * after each sequence, may be NULL).  Outputs, all [.., per value head] so that grouped heads
 * never write the same row: dqh, dkh [T, HO, K] (gradients of the raw q, k rows as used by
 * head h; the caller sums each group), dv [T, HO, V], dg, dbeta [T, HO], ds0 [N, HO, K, V]
 * (may be NULL).  For each token, in reverse, with S_prev the state entering it:
 *     S' = a S_prev, a = exp(g);  x = S'^T k;  u = beta (v - x);  S = S' + k u^T;  o = scale S^T q
 *   dS += scale q do^T;   dq = scale S do
 *   dk = dS u;  du = dS^T k;  dbeta = du . (v - x);  dv = beta du;  dx = -beta du
 *   dS' = dS + k dx^T;  dk += S' dx;  dg = a <dS', S_prev>;  dS = a dS'
 * then through the L2 norm: for y = x / sqrt(|x|^2 + eps), dx = r dy - r^3 (x . dy) x.
 * States are recomputed forward within 64-token segments from stored segment entries.
 * ------------------------------------------------------------------------------------------ */
typedef struct {
    const oracle_job *F;  /* forward description (inputs, shapes, s0) */
    const double *do_;
    const double *dfinal;
    double *dqh, *dkh, *dv, *dg, *dbeta, *ds0;
    int64_t next_unit;
    pthread_mutex_t lock;
} bwd_job;

static void norm_bwd(const double *raw, const double *dy, double *dx, int n, int on) {
    if (!on) {
        for (int d = 0; d < n; ++d) dx[d] = dy[d];
        return;
    }
    double ss = 0.0, dot = 0.0;
    for (int d = 0; d < n; ++d) ss += raw[d] * raw[d];
    const double r = 1.0 / sqrt(ss + 1e-6);
    for (int d = 0; d < n; ++d) dot += raw[d] * dy[d];
    for (int d = 0; d < n; ++d) dx[d] = r * dy[d] - r * r * r * dot * raw[d];
}

static void bwd_unit(const bwd_job *B, int i, int h) {
    const oracle_job *J = B->F;
    const int K = J->K, V = J->V, HO = J->HV, HK = J->HK;
    const int hk = h / (J->HV / J->HK);
    const int64_t t0 = J->cu[i], t1 = J->cu[i + 1], L = t1 - t0;
    const int64_t unit = (int64_t)i * HO + h;
    const int64_t KV = (int64_t)K * V;
    const int SEG = 64;
    const int64_t nseg = (L + SEG - 1) / SEG;

    double *seg = malloc(sizeof(double) * (size_t)((nseg > 0 ? nseg : 1) * KV));
    double *St = malloc(sizeof(double) * (size_t)((SEG + 1) * KV));  /* states within a segment */
    double *S = calloc((size_t)KV, sizeof(double));
    double *dS = calloc((size_t)KV, sizeof(double));
    double *Sp = malloc(sizeof(double) * (size_t)KV);
    double *kn = malloc(sizeof(double) * K), *qn = malloc(sizeof(double) * K);
    double *x = malloc(sizeof(double) * V), *u = malloc(sizeof(double) * V), *du = malloc(sizeof(double) * V);
    double *dx = malloc(sizeof(double) * V);
    double *dkn = malloc(sizeof(double) * K), *dqn = malloc(sizeof(double) * K);
    if (J->s0) memcpy(S, J->s0 + unit * KV, sizeof(double) * (size_t)KV);
    if (B->dfinal) memcpy(dS, B->dfinal + unit * KV, sizeof(double) * (size_t)KV);

    /* one forward step from state P (entering token t) into Q; also returns k_hat, q_hat, x, u */
#define STEP(P, Q, t)                                                                          \
    do {                                                                                       \
        memcpy(qn, J->q + ((t) * HK + hk) * K, sizeof(double) * K);                            \
        memcpy(kn, J->k + ((t) * HK + hk) * K, sizeof(double) * K);                            \
        if (J->l2norm) { l2_normalise(qn, K, 0); l2_normalise(kn, K, 0); }                    \
        const double a_ = exp(J->g[(t) * HO + h]), b_ = J->beta[(t) * HO + h];                 \
        const double *vt_ = J->v + ((t) * J->HV + h) * V;                                      \
        for (int c = 0; c < V; ++c) x[c] = 0.0;                                                \
        for (int r = 0; r < K; ++r)                                                            \
            for (int c = 0; c < V; ++c) x[c] += a_ * (P)[r * V + c] * kn[r];                   \
        for (int c = 0; c < V; ++c) u[c] = b_ * (vt_[c] - x[c]);                               \
        for (int r = 0; r < K; ++r)                                                            \
            for (int c = 0; c < V; ++c) (Q)[r * V + c] = a_ * (P)[r * V + c] + kn[r] * u[c];   \
    } while (0)

    /* forward: segment entry states */
    for (int64_t s = 0; s < nseg; ++s) {
        memcpy(seg + s * KV, S, sizeof(double) * (size_t)KV);
        const int64_t e = (s + 1) * SEG < L ? (s + 1) * SEG : L;
        for (int64_t o = s * SEG; o < e; ++o) {
            STEP(S, Sp, t0 + o);
            memcpy(S, Sp, sizeof(double) * (size_t)KV);
        }
    }
    /* reverse */
    for (int64_t s = nseg - 1; s >= 0; --s) {
        const int64_t b0 = s * SEG, e = (s + 1) * SEG < L ? (s + 1) * SEG : L;
        memcpy(St, seg + s * KV, sizeof(double) * (size_t)KV);
        for (int64_t o = b0; o < e; ++o) STEP(St + (o - b0) * KV, St + (o - b0 + 1) * KV, t0 + o);
        for (int64_t o = e - 1; o >= b0; --o) {
            const int64_t t = t0 + o;
            const double *Sprev = St + (o - b0) * KV, *Snew = St + (o - b0 + 1) * KV;
            STEP(Sprev, Sp, t); /* recomputes k_hat, q_hat, x, u (Sp == Snew) */
            const double a = exp(J->g[t * HO + h]), b = J->beta[t * HO + h];
            const double *vt = J->v + (t * J->HV + h) * V;
            const double *dot = B->do_ + (t * HO + h) * V;
            /* o = scale S^T q */
            for (int r = 0; r < K; ++r) {
                double acc = 0.0;
                for (int c = 0; c < V; ++c) {
                    dS[r * V + c] += J->scale * qn[r] * dot[c];
                    acc += Snew[r * V + c] * dot[c];
                }
                dqn[r] = J->scale * acc;
            }
            /* S = S' + k u^T */
            for (int r = 0; r < K; ++r) {
                double acc = 0.0;
                for (int c = 0; c < V; ++c) acc += dS[r * V + c] * u[c];
                dkn[r] = acc;
            }
            double db = 0.0;
            for (int c = 0; c < V; ++c) {
                double acc = 0.0;
                for (int r = 0; r < K; ++r) acc += dS[r * V + c] * kn[r];
                du[c] = acc;
                db += acc * (vt[c] - x[c]);
                B->dv[(t * HO + h) * V + c] = b * acc;
                dx[c] = -b * acc;
            }
            B->dbeta[t * HO + h] = db;
            /* x = S'^T k, S' = a S_prev */
            double da = 0.0;
            for (int r = 0; r < K; ++r) {
                double acc = 0.0;
                for (int c = 0; c < V; ++c) {
                    const double sp = a * Sprev[r * V + c];
                    acc += sp * dx[c];
                    double dsp = dS[r * V + c] + kn[r] * dx[c];
                    if (J->mutation == 14) dsp = dS[r * V + c]; /* planted: decay gradient misses the erase path */
                    da += dsp * Sprev[r * V + c];
                    dS[r * V + c] = a * (dS[r * V + c] + kn[r] * dx[c]);
                }
                if (J->mutation != 15) dkn[r] += acc; /* planted (15): k misses the S' dx term */
            }
            B->dg[t * HO + h] = da * a;
            norm_bwd(J->q + (t * HK + hk) * K, dqn, B->dqh + (t * HO + h) * K, K, J->l2norm);
            norm_bwd(J->k + (t * HK + hk) * K, dkn, B->dkh + (t * HO + h) * K, K, J->l2norm);
        }
    }
#undef STEP
    if (B->ds0) memcpy(B->ds0 + unit * KV, dS, sizeof(double) * (size_t)KV);
    free(seg); free(St); free(S); free(dS); free(Sp); free(kn); free(qn);
    free(x); free(u); free(du); free(dx); free(dkn); free(dqn);
}

static void *bwd_worker(void *arg) {
    bwd_job *B = (bwd_job *)arg;
    const oracle_job *J = B->F;
    const int64_t units = (int64_t)J->N * J->HV;
    for (;;) {
        pthread_mutex_lock(&B->lock);
        int64_t u = B->next_unit++;
        pthread_mutex_unlock(&B->lock);
        if (u >= units) break;
        if (J->unit_mask && !J->unit_mask[u]) continue;
        bwd_unit(B, (int)(u / J->HV), (int)(u % J->HV));
    }
    return NULL;
}

int gdn_oracle_bwd(const double *q, const double *k, const double *v,
                   const double *g, const double *beta, const int64_t *cu,
                   int64_t T, int N, int HK, int HV, int K, int V,
                   double scale, int l2norm, const double *s0,
                   const double *do_, const double *dfinal,
                   double *dqh, double *dkh, double *dv, double *dg, double *dbeta, double *ds0,
                   const unsigned char *unit_mask, int nthreads, int mutation) {
    if (N < 0 || HK <= 0 || HV <= 0 || HV % HK != 0 || K <= 0 || V <= 0) return -1;
    if (cu[0] != 0 || cu[N] != T) return -1;
    for (int i = 0; i < N; ++i)
        if (cu[i + 1] < cu[i]) return -1;
    oracle_job J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.cu = cu;
    J.T = T; J.N = N; J.HK = HK; J.HV = HV; J.K = K; J.V = V;
    J.scale = scale; J.l2norm = l2norm; J.s0 = s0; J.unit_mask = unit_mask; J.mutation = mutation;
    bwd_job B;
    memset(&B, 0, sizeof(B));
    B.F = &J; B.do_ = do_; B.dfinal = dfinal;
    B.dqh = dqh; B.dkh = dkh; B.dv = dv; B.dg = dg; B.dbeta = dbeta; B.ds0 = ds0;
    pthread_mutex_init(&B.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    pthread_t *th = malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, bwd_worker, &B);
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(th);
    pthread_mutex_destroy(&B.lock);
    return 0;
}
