/*
 * kda_oracle_bwd.c -- plain fp64 CPU oracle for the gradient of the KDA forward pass.
 * TEST INFRASTRUCTURE ONLY: the product path never links, loads or calls this file; only
 * the tests and the CPU baseline leg of the benchmark do.
 *
 * What it computes.  FlashKDA's README ("Kernel API") defines a forward pass only; its
 * gradient is fixed by that definition.  For every sequence n and head h the forward
 * recurrence (the same one kda_oracle.c runs, here on fp64 inputs) is
 *     alpha_t = exp(ghat_t),  beta_t = sigmoid(b_t),  qh_t = q_t / sqrt(|q_t|^2 + 1e-6),
 *     kh_t = k_t / sqrt(|k_t|^2 + 1e-6),
 *     P_t = Diag(alpha_t) S_{t-1},   u_t = v_t - P_t^T kh_t,
 *     S_t = P_t + beta_t kh_t u_t^T,  o_t = scale S_t^T qh_t,
 * with the gate ghat of kda_oracle.c (safe sigmoid gate, softplus gate or a pre-activated
 * g) and its switches.  Given dO = dL/do_t for every token and dF = dL/dS_final (or zero),
 * this file returns dL/dq, dL/dk, dL/dv, dL/dg, dL/db (the beta logits), dL/dS_0 and the
 * parameter gradients dL/dA_log[h] and dL/ddt_bias[h, :] (summed over all tokens of all
 * sequences), by running the recurrence forward once, keeping every state, and then
 * applying the chain rule to each step in reverse:
 *     dS_t += scale qh_t dO_t^T;            dqh_t = scale S_t dO_t
 *     w_t = dS_t^T kh_t;  du_t = beta_t w_t;  dv_t = du_t;  dbeta_t = u_t . w_t
 *     dkh_t = beta_t dS_t u_t - P_t du_t
 *     dP_t = dS_t - kh_t du_t^T;  dalpha_t[c] = sum_j dP_t[c][j] S_{t-1}[c][j]
 *     dS_{t-1} = Diag(alpha_t) dP_t
 * then through the normalisation (dq = (dqh - qh (qh . dqh)) / sqrt(|q|^2 + 1e-6)), the
 * beta sigmoid (db = dbeta beta (1 - beta)) and the gate (dghat = dalpha alpha, then the
 * derivative of the gate formula with respect to g, dt_bias and A_log).
 *
 * Everything is fp64, with plain loops; states are kept whole for every token of a
 * sequence (T_seq x K x V doubles per worker thread).  The gradient is pinned against
 * central finite differences of kda_oracle_fwd64 (the same forward on fp64 inputs), whose
 * outputs are in turn pinned to kda_oracle_fwd on bf16-exact inputs.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { BW_GATE_PREACTIVATED = 1, BW_BETA_PREACTIVATED = 2, BW_NO_QK_L2NORM = 4, BW_GATE_SOFTPLUS = 8 };

static double bw_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }
static double bw_softplus(double x) { return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x)); }

typedef struct {
    int64_t B, T, H, K, V, N;
    int flags;
    const double *q, *k, *v, *g, *beta;
    double scale, lower_bound;
    const double *A_log, *dt_bias;
    const double *initial_state;
    const int64_t *cu_seqlens;
    const double *dout, *dfinal;       /* backward only; dfinal may be NULL */
    double *out, *final_state;         /* forward results, may be NULL */
    double *dq, *dk, *dv, *dg, *dbeta, *dh0;
    double *dA_pair, *ddt_pair;        /* [N*H] and [N*H*K]: per-pair parameter gradients */
    int backward;
    int64_t next_pair;
    pthread_mutex_t lock;
} bw_job;

typedef struct {
    double *S;      /* states S_0..S_len, each K x V (row c, column j) */
    double *alpha, *qh, *kh, *u;  /* per token: K, K, K, V */
    double *beta;   /* per token */
    double *rq, *rk;
    double *dS, *dP, *w, *du, *dqh, *dkh, *dal;
    int64_t cap;    /* tokens the buffers hold */
} bw_ws;

static void bw_ws_free(bw_ws *W) {
    free(W->S); free(W->alpha); free(W->qh); free(W->kh); free(W->u); free(W->beta);
    free(W->rq); free(W->rk); free(W->dS); free(W->dP); free(W->w); free(W->du);
    free(W->dqh); free(W->dkh); free(W->dal);
    memset(W, 0, sizeof *W);
}

static int bw_ws_reserve(bw_ws *W, int64_t len, int64_t K, int64_t V) {
    if (len <= W->cap && W->S) return 0;
    bw_ws_free(W);
    const size_t L = (size_t)(len > 0 ? len : 1);
    W->S = (double *)malloc(sizeof(double) * (L + 1) * (size_t)(K * V));
    W->alpha = (double *)malloc(sizeof(double) * L * (size_t)K);
    W->qh = (double *)malloc(sizeof(double) * L * (size_t)K);
    W->kh = (double *)malloc(sizeof(double) * L * (size_t)K);
    W->u = (double *)malloc(sizeof(double) * L * (size_t)V);
    W->beta = (double *)malloc(sizeof(double) * L);
    W->rq = (double *)malloc(sizeof(double) * L);
    W->rk = (double *)malloc(sizeof(double) * L);
    W->dS = (double *)malloc(sizeof(double) * (size_t)(K * V));
    W->dP = (double *)malloc(sizeof(double) * (size_t)(K * V));
    W->w = (double *)malloc(sizeof(double) * (size_t)V);
    W->du = (double *)malloc(sizeof(double) * (size_t)V);
    W->dqh = (double *)malloc(sizeof(double) * (size_t)K);
    W->dkh = (double *)malloc(sizeof(double) * (size_t)K);
    W->dal = (double *)malloc(sizeof(double) * (size_t)K);
    W->cap = (int64_t)L;
    if (!W->S || !W->alpha || !W->qh || !W->kh || !W->u || !W->beta || !W->rq || !W->rk || !W->dS ||
        !W->dP || !W->w || !W->du || !W->dqh || !W->dkh || !W->dal) {
        bw_ws_free(W);
        return -1;
    }
    return 0;
}

/* The gate's pre-activation x = g + dt_bias and its decay; ghat is the natural-log decay. */
static double bw_ghat(const bw_job *J, int64_t h, double gval, int64_t c, double rate) {
    if (J->flags & BW_GATE_PREACTIVATED) return gval;
    const double x = gval + J->dt_bias[h * J->K + c];
    if (J->flags & BW_GATE_SOFTPLUS) return -rate * bw_softplus(x);
    return J->lower_bound * bw_sigmoid(rate * x);
}

static int bw_run_pair(bw_job *J, int64_t n, int64_t h, bw_ws *W) {
    const int64_t H = J->H, K = J->K, V = J->V, KV = K * V;
    int64_t t0, t1;
    if (J->cu_seqlens) {
        t0 = J->cu_seqlens[n];
        t1 = J->cu_seqlens[n + 1];
    } else {
        t0 = n * J->T;
        t1 = t0 + J->T;
    }
    const int64_t len = t1 - t0;
    if (bw_ws_reserve(W, len, K, V)) return -1;
    const int norm = !(J->flags & BW_NO_QK_L2NORM);
    const double rate = (J->flags & BW_GATE_PREACTIVATED) ? 0.0 : exp(J->A_log[h]);

    /* ---- forward, keeping S_0 .. S_len */
    double *S0 = W->S;
    if (J->initial_state) {
        const double *s0 = J->initial_state + (n * H + h) * V * K;
        for (int64_t c = 0; c < K; ++c)
            for (int64_t j = 0; j < V; ++j) S0[c * V + j] = s0[j * K + c];
    } else {
        memset(S0, 0, sizeof(double) * (size_t)KV);
    }
    for (int64_t i = 0; i < len; ++i) {
        const int64_t t = t0 + i;
        const double *qt = J->q + (t * H + h) * K, *kt = J->k + (t * H + h) * K;
        const double *gt = J->g + (t * H + h) * K, *vt = J->v + (t * H + h) * V;
        double *al = W->alpha + i * K, *qh = W->qh + i * K, *kh = W->kh + i * K, *u = W->u + i * V;
        double qq = 0.0, kk = 0.0;
        for (int64_t c = 0; c < K; ++c) {
            qq += qt[c] * qt[c];
            kk += kt[c] * kt[c];
        }
        W->rq[i] = norm ? 1.0 / sqrt(qq + 1e-6) : 1.0;
        W->rk[i] = norm ? 1.0 / sqrt(kk + 1e-6) : 1.0;
        for (int64_t c = 0; c < K; ++c) {
            qh[c] = qt[c] * W->rq[i];
            kh[c] = kt[c] * W->rk[i];
            al[c] = exp(bw_ghat(J, h, gt[c], c, rate));
        }
        const double braw = J->beta[t * H + h];
        const double b = (J->flags & BW_BETA_PREACTIVATED) ? braw : bw_sigmoid(braw);
        W->beta[i] = b;
        const double *Sp = W->S + i * KV;
        double *Sn = W->S + (i + 1) * KV;
        /* P = Diag(alpha) S_{t-1}; u = v - P^T kh; S_t = P + beta kh u^T */
        for (int64_t c = 0; c < K; ++c)
            for (int64_t j = 0; j < V; ++j) Sn[c * V + j] = al[c] * Sp[c * V + j];
        for (int64_t j = 0; j < V; ++j) {
            double s = 0.0;
            for (int64_t c = 0; c < K; ++c) s += Sn[c * V + j] * kh[c];
            u[j] = vt[j] - s;
        }
        for (int64_t c = 0; c < K; ++c)
            for (int64_t j = 0; j < V; ++j) Sn[c * V + j] += b * kh[c] * u[j];
        if (J->out) {
            double *o = J->out + (t * H + h) * V;
            for (int64_t j = 0; j < V; ++j) {
                double s = 0.0;
                for (int64_t c = 0; c < K; ++c) s += Sn[c * V + j] * qh[c];
                o[j] = J->scale * s;
            }
        }
    }
    if (J->final_state) {
        const double *Sf = W->S + len * KV;
        double *sf = J->final_state + (n * H + h) * V * K;
        for (int64_t c = 0; c < K; ++c)
            for (int64_t j = 0; j < V; ++j) sf[j * K + c] = Sf[c * V + j];
    }
    if (!J->backward) return 0;

    /* ---- reverse */
    double *dS = W->dS, *dP = W->dP;
    if (J->dfinal) {
        const double *df = J->dfinal + (n * H + h) * V * K;
        for (int64_t c = 0; c < K; ++c)
            for (int64_t j = 0; j < V; ++j) dS[c * V + j] = df[j * K + c];
    } else {
        memset(dS, 0, sizeof(double) * (size_t)KV);
    }
    double dA = 0.0;
    double *ddt = J->ddt_pair + (n * H + h) * K;
    for (int64_t c = 0; c < K; ++c) ddt[c] = 0.0;
    for (int64_t i = len - 1; i >= 0; --i) {
        const int64_t t = t0 + i;
        const double *al = W->alpha + i * K, *qh = W->qh + i * K, *kh = W->kh + i * K, *u = W->u + i * V;
        const double b = W->beta[i];
        const double *Sprev = W->S + i * KV, *St = W->S + (i + 1) * KV;
        const double *dO = J->dout + (t * H + h) * V;
        /* output: o = scale S_t^T qh */
        for (int64_t c = 0; c < K; ++c) {
            double s = 0.0;
            for (int64_t j = 0; j < V; ++j) s += St[c * V + j] * dO[j];
            W->dqh[c] = J->scale * s;
        }
        for (int64_t c = 0; c < K; ++c)
            for (int64_t j = 0; j < V; ++j) dS[c * V + j] += J->scale * qh[c] * dO[j];
        /* S_t = P + beta kh u^T */
        double dbeta = 0.0;
        for (int64_t j = 0; j < V; ++j) {
            double s = 0.0;
            for (int64_t c = 0; c < K; ++c) s += dS[c * V + j] * kh[c];
            W->w[j] = s;
            W->du[j] = b * s;
            dbeta += u[j] * s;
            J->dv[(t * H + h) * V + j] = W->du[j];
        }
        /* dkh = beta dS u - P du, with P = Diag(alpha) S_{t-1} */
        for (int64_t c = 0; c < K; ++c) {
            double s1 = 0.0, s2 = 0.0;
            for (int64_t j = 0; j < V; ++j) {
                s1 += dS[c * V + j] * u[j];
                s2 += al[c] * Sprev[c * V + j] * W->du[j];
            }
            W->dkh[c] = b * s1 - s2;
        }
        /* dP = dS - kh du^T (the u = v - P^T kh path); dalpha; dS_{t-1} = Diag(alpha) dP */
        for (int64_t c = 0; c < K; ++c) {
            double s = 0.0;
            for (int64_t j = 0; j < V; ++j) {
                dP[c * V + j] = dS[c * V + j] - kh[c] * W->du[j];
                s += dP[c * V + j] * Sprev[c * V + j];
            }
            W->dal[c] = s;
            for (int64_t j = 0; j < V; ++j) dS[c * V + j] = al[c] * dP[c * V + j];
        }
        /* through the normalisations */
        double qd = 0.0, kd = 0.0;
        for (int64_t c = 0; c < K; ++c) {
            qd += qh[c] * W->dqh[c];
            kd += kh[c] * W->dkh[c];
        }
        for (int64_t c = 0; c < K; ++c) {
            J->dq[(t * H + h) * K + c] = norm ? W->rq[i] * (W->dqh[c] - qh[c] * qd) : W->dqh[c];
            J->dk[(t * H + h) * K + c] = norm ? W->rk[i] * (W->dkh[c] - kh[c] * kd) : W->dkh[c];
        }
        /* beta */
        J->dbeta[t * H + h] = (J->flags & BW_BETA_PREACTIVATED) ? dbeta : dbeta * b * (1.0 - b);
        /* gate: dghat = dalpha alpha */
        const double *gt = J->g + (t * H + h) * K;
        for (int64_t c = 0; c < K; ++c) {
            const double dgh = W->dal[c] * al[c];
            double dgv;
            if (J->flags & BW_GATE_PREACTIVATED) {
                dgv = dgh;
            } else if (J->flags & BW_GATE_SOFTPLUS) {
                /* ghat = -rate softplus(x): d/dx = -rate sigmoid(x), d/dA_log = ghat */
                const double x = gt[c] + J->dt_bias[h * K + c];
                dgv = dgh * (-rate * bw_sigmoid(x));
                dA += dgh * (-rate * bw_softplus(x));
                ddt[c] += dgv;
            } else {
                /* ghat = lb sigmoid(z), z = rate x: d/dx = lb s(1-s) rate, d/dA_log = lb s(1-s) z */
                const double x = gt[c] + J->dt_bias[h * K + c];
                const double z = rate * x, s = bw_sigmoid(z);
                const double dz = dgh * J->lower_bound * s * (1.0 - s);
                dgv = dz * rate;
                dA += dz * z;
                ddt[c] += dgv;
            }
            J->dg[(t * H + h) * K + c] = dgv;
        }
    }
    J->dA_pair[n * H + h] = dA;
    if (J->dh0) {
        double *d0 = J->dh0 + (n * H + h) * V * K;
        for (int64_t c = 0; c < K; ++c)
            for (int64_t j = 0; j < V; ++j) d0[j * K + c] = dS[c * V + j];
    }
    return 0;
}

static void *bw_worker(void *arg) {
    bw_job *J = (bw_job *)arg;
    bw_ws W;
    memset(&W, 0, sizeof W);
    void *rc = NULL;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int64_t p = J->next_pair++;
        pthread_mutex_unlock(&J->lock);
        if (p >= J->N * J->H) break;
        if (bw_run_pair(J, p / J->H, p % J->H, &W)) {
            rc = (void *)1;
            break;
        }
    }
    bw_ws_free(&W);
    return rc;
}

static int bw_run(bw_job *J, int nthreads) {
    int64_t pairs = J->N * J->H;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > pairs) nthreads = (int)(pairs > 0 ? pairs : 1);
    J->next_pair = 0;
    pthread_mutex_init(&J->lock, NULL);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th) return -2;
    int started = 0, rc = 0;
    for (int i = 0; i < nthreads; ++i)
        if (pthread_create(&th[i], NULL, bw_worker, J) == 0) ++started;
    if (started == 0) rc = (bw_worker(J) == NULL) ? 0 : -2;
    for (int i = 0; i < started; ++i) {
        void *r = NULL;
        pthread_join(th[i], &r);
        if (r != NULL) rc = -2;
    }
    free(th);
    pthread_mutex_destroy(&J->lock);
    return rc;
}

static int bw_check(int64_t B, int64_t T, int64_t H, int64_t K, int64_t V, int64_t N, int flags,
                    const int64_t *cu_seqlens) {
    if (B < 0 || T < 0 || H <= 0 || K <= 0 || V <= 0 || N < 0) return -1;
    if (!cu_seqlens && N != B) return -1;
    if (cu_seqlens && B != 1) return -1;
    if ((flags & BW_GATE_PREACTIVATED) && (flags & BW_GATE_SOFTPLUS)) return -1;
    return 0;
}

/*
 * The forward recurrence on fp64 inputs (q, k, g [B,T,H,K]; v [B,T,H,V]; beta [B,T,H] logits;
 * A_log [H]; dt_bias [H,K]; initial_state [N,H,V,K] or NULL): writes out [B,T,H,V] and, if
 * given, final_state [N,H,V,K].  Returns 0, -1 (bad argument) or -2 (allocation failure).
 */
int kda_oracle_fwd64(int64_t B, int64_t T, int64_t H, int64_t K, int64_t V, int64_t N, int flags,
                     const double *q, const double *k, const double *v, const double *g, const double *beta,
                     double scale, const double *A_log, const double *dt_bias, double lower_bound,
                     const double *initial_state, const int64_t *cu_seqlens, double *out,
                     double *final_state, int nthreads) {
    if (bw_check(B, T, H, K, V, N, flags, cu_seqlens)) return -1;
    bw_job J;
    memset(&J, 0, sizeof J);
    J.B = B; J.T = T; J.H = H; J.K = K; J.V = V; J.N = N; J.flags = flags;
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta;
    J.scale = scale; J.lower_bound = lower_bound; J.A_log = A_log; J.dt_bias = dt_bias;
    J.initial_state = initial_state; J.cu_seqlens = cu_seqlens;
    J.out = out; J.final_state = final_state;
    J.backward = 0;
    return bw_run(&J, nthreads);
}

/*
 * The gradient: inputs as kda_oracle_fwd64 plus dout [B,T,H,V] and dfinal [N,H,V,K] (or NULL:
 * the final state does not enter the loss).  Writes dq, dk, dg [B,T,H,K], dv [B,T,H,V],
 * dbeta [B,T,H] (with respect to the beta logits, or to beta itself when it is
 * pre-activated), dh0 [N,H,V,K] (if not NULL), and dA_log [H], ddt_bias [H,K] (zero for a
 * pre-activated gate).  Returns 0, -1 or -2.
 */
int kda_oracle_bwd(int64_t B, int64_t T, int64_t H, int64_t K, int64_t V, int64_t N, int flags,
                   const double *q, const double *k, const double *v, const double *g, const double *beta,
                   double scale, const double *A_log, const double *dt_bias, double lower_bound,
                   const double *initial_state, const int64_t *cu_seqlens, const double *dout,
                   const double *dfinal, double *dq, double *dk, double *dv, double *dg, double *dbeta,
                   double *dh0, double *dA_log, double *ddt_bias, int nthreads) {
    if (bw_check(B, T, H, K, V, N, flags, cu_seqlens)) return -1;
    if (!dout || !dq || !dk || !dv || !dg || !dbeta || !dA_log || !ddt_bias) return -1;
    bw_job J;
    memset(&J, 0, sizeof J);
    J.B = B; J.T = T; J.H = H; J.K = K; J.V = V; J.N = N; J.flags = flags;
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta;
    J.scale = scale; J.lower_bound = lower_bound; J.A_log = A_log; J.dt_bias = dt_bias;
    J.initial_state = initial_state; J.cu_seqlens = cu_seqlens;
    J.dout = dout; J.dfinal = dfinal;
    J.dq = dq; J.dk = dk; J.dv = dv; J.dg = dg; J.dbeta = dbeta; J.dh0 = dh0;
    J.backward = 1;
    const size_t pairs = (size_t)(N * H);
    J.dA_pair = (double *)calloc(pairs > 0 ? pairs : 1, sizeof(double));
    J.ddt_pair = (double *)calloc((pairs > 0 ? pairs : 1) * (size_t)K, sizeof(double));
    if (!J.dA_pair || !J.ddt_pair) {
        free(J.dA_pair);
        free(J.ddt_pair);
        return -2;
    }
    const int rc = bw_run(&J, nthreads);
    /* parameter gradients: sum over sequences in order */
    for (int64_t h = 0; h < H; ++h) {
        double a = 0.0;
        for (int64_t n = 0; n < N; ++n) a += J.dA_pair[n * H + h];
        dA_log[h] = a;
        for (int64_t c = 0; c < K; ++c) {
            double s = 0.0;
            for (int64_t n = 0; n < N; ++n) s += J.ddt_pair[(n * H + h) * K + c];
            ddt_bias[h * K + c] = s;
        }
    }
    free(J.dA_pair);
    free(J.ddt_pair);
    return rc;
}
