/*
 * kda_oracle.c -- float64 CPU oracle for Kimi Delta Attention (KDA).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plainly written
 * definition that the CUDA library is checked against.  Only the test suite,
 * the smoke check and the CPU-baseline leg of the benchmark may load it.  It
 * shares no code, header or constant with the CUDA path.
 *
 * What it computes (all in float64):
 *
 *   Per head, with the state S (K x V) and per token t:
 *       a_t  = exp(max(g_t, -5))                      (per key channel)
 *       P_t  = diag(a_t) S_{t-1}                       (decay first)
 *       e_t  = v_t - P_t^T k_t                         (key reads the decayed state)
 *       S_t  = P_t + beta_t k_t e_t^T                  (delta-rule write)
 *       o_t  = S_t^T (scale q_t)                       (query reads the updated state)
 *
 *   Sources:
 *     - "KDA 训练 → 推理 手写实现" (K3 README), table 实现路线表, row L1:
 *       the recurrence S_t = exp(g_t)*S + (beta_t k_t)(v_t - k_t.S), o_t = (q_t scale) S.
 *     - "KDA CUDA Trainer" README, section on the sequence-mixing module:
 *       a per-key forget gate decays the state, then the key-prediction
 *       error is written back, and queries read the UPDATED state.
 *     - K3 README, table 关键约束 / 风险点: GVA (q/k repeated over
 *       G = HV/H with repeat_interleave, so value head hv uses key head
 *       hv / G; dq/dk summed back over the group), scale 1/sqrt(K) applied to
 *       q at entry, g clamped before exp with lower bound -5.
 *
 *   Readings taken where the pages are open:
 *     - k reads the decayed state diag(a_t) S_{t-1} (the row-L1 formula
 *       applies exp(g) first and then writes "k_t.S" of that product).
 *     - beta is one scalar per token and value head, used as given.
 *     - d max(g,-5)/dg = 1 where g >= -5 (inclusive), else 0.
 *
 * Functions:
 *   kda_oracle_fwd_recurrent   token-by-token forward (row L1).
 *   kda_oracle_bwd_recurrent   hand-derived reverse-time backward (row L1:
 *                              dq, dk, dv, dg, dbeta, and dh0).
 *   kda_oracle_fwd_chunked     the chunk form of K3 row L2: (1) cumsum of
 *                              the clamped gate inside each chunk, (2) the
 *                              lower-triangular system, (3) its solve,
 *                              (4) the state passed between chunks.
 *   kda_oracle_chunk_wy        the row-L2 quantities of one chunk (A, T, W,
 *                              U, Aqk), exposed for the WY pins.
 *   kda_oracle_step            one decode token applied in place (row L6,
 *                              state [B,HV,K,V]).
 *   kda_oracle_l2norm(_bwd)    x / max(||x||, 1e-12) per row and its
 *                              backward (the q/k L2-norm variant).
 *
 * Layouts (row-major, contiguous):
 *   q, k      [B,T,H,K]     v, o   [B,T,HV,V]     g  [B,T,HV,K]
 *   beta      [B,T,HV]      states [B,HV,K,V]
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int B, T, H, HV, K, V;
    double scale;
} odims;

static double gate_hat(double g) { return g < -5.0 ? -5.0 : g; }

static size_t ix_qk(const odims* d, int b, int t, int h, int c) {
    return (((size_t)b * d->T + t) * d->H + h) * d->K + c;
}
static size_t ix_v(const odims* d, int b, int t, int hv, int j) {
    return (((size_t)b * d->T + t) * d->HV + hv) * d->V + j;
}
static size_t ix_g(const odims* d, int b, int t, int hv, int c) {
    return (((size_t)b * d->T + t) * d->HV + hv) * d->K + c;
}
static size_t ix_beta(const odims* d, int b, int t, int hv) {
    return ((size_t)b * d->T + t) * d->HV + hv;
}
static size_t ix_state(const odims* d, int b, int hv) {
    return ((size_t)b * d->HV + hv) * (size_t)d->K * d->V;
}

int kda_oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* One token of the recurrence on state S (K x V), in place.  o (V) may be
 * NULL.  Optional outputs: P (decayed state, K x V) and e (V). */
static void token_step(int K, int V, double scale, const double* q, const double* k,
                       const double* v, const double* g, double beta, double* S,
                       double* o, double* e_out) {
    double e[V > 0 ? V : 1];
    for (int c = 0; c < K; ++c) {
        double a = exp(gate_hat(g[c]));
        for (int j = 0; j < V; ++j) S[(size_t)c * V + j] *= a; /* S now holds P_t */
    }
    for (int j = 0; j < V; ++j) {
        double acc = 0.0;
        for (int c = 0; c < K; ++c) acc += k[c] * S[(size_t)c * V + j];
        e[j] = v[j] - acc;
    }
    for (int c = 0; c < K; ++c) {
        double bk = beta * k[c];
        for (int j = 0; j < V; ++j) S[(size_t)c * V + j] += bk * e[j];
    }
    if (o) {
        for (int j = 0; j < V; ++j) {
            double acc = 0.0;
            for (int c = 0; c < K; ++c) acc += scale * q[c] * S[(size_t)c * V + j];
            o[j] = acc;
        }
    }
    if (e_out)
        for (int j = 0; j < V; ++j) e_out[j] = e[j];
}

/* Gather the per-token vectors of one head into small contiguous buffers. */
static void gather_token(const odims* d, int b, int t, int hv, const double* q,
                         const double* k, const double* v, const double* g, const double* beta,
                         double* qt, double* kt, double* vt, double* gt, double* bt) {
    int h = hv / (d->HV / d->H);
    for (int c = 0; c < d->K; ++c) {
        qt[c] = q[ix_qk(d, b, t, h, c)];
        kt[c] = k[ix_qk(d, b, t, h, c)];
        gt[c] = g[ix_g(d, b, t, hv, c)];
    }
    for (int j = 0; j < d->V; ++j) vt[j] = v[ix_v(d, b, t, hv, j)];
    *bt = beta[ix_beta(d, b, t, hv)];
}

/* ------------------------------------------------------------------------ */
/* Forward, token by token.                                                  */
/* ------------------------------------------------------------------------ */
void kda_oracle_fwd_recurrent(int B, int T, int H, int HV, int K, int V, double scale,
                              const double* q, const double* k, const double* v,
                              const double* g, const double* beta, const double* h0,
                              double* o, double* ht) {
    odims d = {B, T, H, HV, K, V, scale};
    int nheads = B * HV;
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < nheads; ++bh) {
        int b = bh / HV, hv = bh % HV;
        size_t KV = (size_t)K * V;
        double* S = (double*)calloc(KV, sizeof(double));
        double *qt = malloc(K * sizeof(double)), *kt = malloc(K * sizeof(double)),
               *gt = malloc(K * sizeof(double)), *vt = malloc(V * sizeof(double)),
               *ot = malloc(V * sizeof(double));
        double bt;
        if (h0) memcpy(S, h0 + ix_state(&d, b, hv), KV * sizeof(double));
        for (int t = 0; t < T; ++t) {
            gather_token(&d, b, t, hv, q, k, v, g, beta, qt, kt, vt, gt, &bt);
            token_step(K, V, scale, qt, kt, vt, gt, bt, S, ot, NULL);
            for (int j = 0; j < V; ++j) o[ix_v(&d, b, t, hv, j)] = ot[j];
        }
        if (ht) memcpy(ht + ix_state(&d, b, hv), S, KV * sizeof(double));
        free(S); free(qt); free(kt); free(gt); free(vt); free(ot);
    }
}

/* ------------------------------------------------------------------------ */
/* Backward, reverse time.                                                   */
/*                                                                           */
/* Per token, walking t = T-1 .. 0 with dS the gradient w.r.t. S_t:          */
/*   o_t = S_t^T qs          -> dS += qs do^T,     dqs = S_t do              */
/*   S_t = P + beta k e^T    -> dP = dS, dbeta = k^T dS e, dk = beta dS e,   */
/*                              de = beta dS^T k                             */
/*   e = v - P^T k           -> dv = de, dk -= P de, dP -= k de^T            */
/*   P = diag(a) S_{t-1}     -> dg = rowsum(dP o P) [g >= -5],               */
/*                              dS_{t-1} = diag(a) dP                        */
/*   qs = scale q            -> dq = scale dqs                               */
/* The states S_{t-1} are rebuilt by replaying the forward from checkpoints  */
/* taken every SEG tokens.  dq/dk are formed per value head and then summed  */
/* over the G value heads that share a key head.                             */
/* ------------------------------------------------------------------------ */
#define SEG 64

void kda_oracle_bwd_recurrent(int B, int T, int H, int HV, int K, int V, double scale,
                              const double* q, const double* k, const double* v,
                              const double* g, const double* beta, const double* h0,
                              const double* dout, const double* dht, double* dq,
                              double* dk, double* dv, double* dg, double* dbeta,
                              double* dh0) {
    odims d = {B, T, H, HV, K, V, scale};
    int nheads = B * HV;
    int G = HV / H;
    size_t nqk_hv = (size_t)B * T * HV * K;
    /* dq, dk per value head; summed over the group at the end. */
    double* dq_hv = (double*)calloc(nqk_hv, sizeof(double));
    double* dk_hv = (double*)calloc(nqk_hv, sizeof(double));
    int nseg = (T + SEG - 1) / SEG;

#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < nheads; ++bh) {
        int b = bh / HV, hv = bh % HV;
        size_t KV = (size_t)K * V;
        double* ckpt = (double*)calloc((size_t)(nseg > 0 ? nseg : 1) * KV, sizeof(double));
        double* states = (double*)calloc((size_t)(SEG + 1) * KV, sizeof(double));
        double* dS = (double*)calloc(KV, sizeof(double));
        double* P = (double*)calloc(KV, sizeof(double));
        double *qt = malloc(K * sizeof(double)), *kt = malloc(K * sizeof(double)),
               *gt = malloc(K * sizeof(double)), *vt = malloc(V * sizeof(double)),
               *e = malloc(V * sizeof(double)), *de = malloc(V * sizeof(double)),
               *dot = malloc(V * sizeof(double)), *a = malloc(K * sizeof(double)),
               *dkt = malloc(K * sizeof(double)), *dqs = malloc(K * sizeof(double));
        double bt;

        /* forward pass: checkpoint the state before each segment */
        double* S = states; /* scratch */
        memset(S, 0, KV * sizeof(double));
        if (h0) memcpy(S, h0 + ix_state(&d, b, hv), KV * sizeof(double));
        for (int t = 0; t < T; ++t) {
            if (t % SEG == 0) memcpy(ckpt + (size_t)(t / SEG) * KV, S, KV * sizeof(double));
            gather_token(&d, b, t, hv, q, k, v, g, beta, qt, kt, vt, gt, &bt);
            token_step(K, V, scale, qt, kt, vt, gt, bt, S, NULL, NULL);
        }

        if (dht) memcpy(dS, dht + ix_state(&d, b, hv), KV * sizeof(double));

        for (int s = nseg - 1; s >= 0; --s) {
            int t0 = s * SEG, t1 = t0 + SEG < T ? t0 + SEG : T;
            /* replay: states[i] = S_{t0+i-1} (state before token t0+i) */
            memcpy(states, ckpt + (size_t)s * KV, KV * sizeof(double));
            for (int t = t0; t < t1; ++t) {
                double* nxt = states + (size_t)(t - t0 + 1) * KV;
                memcpy(nxt, states + (size_t)(t - t0) * KV, KV * sizeof(double));
                gather_token(&d, b, t, hv, q, k, v, g, beta, qt, kt, vt, gt, &bt);
                token_step(K, V, scale, qt, kt, vt, gt, bt, nxt, NULL, NULL);
            }
            for (int t = t1 - 1; t >= t0; --t) {
                const double* Sprev = states + (size_t)(t - t0) * KV;
                const double* Scur = states + (size_t)(t - t0 + 1) * KV;
                gather_token(&d, b, t, hv, q, k, v, g, beta, qt, kt, vt, gt, &bt);
                for (int j = 0; j < V; ++j) dot[j] = dout[ix_v(&d, b, t, hv, j)];
                for (int c = 0; c < K; ++c) a[c] = exp(gate_hat(gt[c]));
                for (int c = 0; c < K; ++c)
                    for (int j = 0; j < V; ++j) P[(size_t)c * V + j] = a[c] * Sprev[(size_t)c * V + j];
                for (int j = 0; j < V; ++j) {
                    double acc = 0.0;
                    for (int c = 0; c < K; ++c) acc += kt[c] * P[(size_t)c * V + j];
                    e[j] = vt[j] - acc;
                }
                /* output read: o_t = S_t^T (scale q_t) */
                for (int c = 0; c < K; ++c) {
                    double acc = 0.0;
                    for (int j = 0; j < V; ++j) {
                        dS[(size_t)c * V + j] += scale * qt[c] * dot[j];
                        acc += Scur[(size_t)c * V + j] * dot[j];
                    }
                    dqs[c] = acc;
                }
                /* delta-rule write: S_t = P + beta k e^T */
                double db = 0.0;
                for (int c = 0; c < K; ++c) {
                    double acc = 0.0;
                    for (int j = 0; j < V; ++j) acc += dS[(size_t)c * V + j] * e[j];
                    dkt[c] = bt * acc;
                    db += kt[c] * acc;
                }
                for (int j = 0; j < V; ++j) {
                    double acc = 0.0;
                    for (int c = 0; c < K; ++c) acc += dS[(size_t)c * V + j] * kt[c];
                    de[j] = bt * acc;
                }
                /* error: e = v - P^T k ; dP = dS - k de^T */
                for (int c = 0; c < K; ++c) {
                    double acc = 0.0;
                    for (int j = 0; j < V; ++j) acc += P[(size_t)c * V + j] * de[j];
                    dkt[c] -= acc;
                }
                /* decay: P = diag(a) S_{t-1} */
                for (int c = 0; c < K; ++c) {
                    double acc = 0.0;
                    for (int j = 0; j < V; ++j) {
                        double dP = dS[(size_t)c * V + j] - kt[c] * de[j];
                        acc += dP * P[(size_t)c * V + j];
                        dS[(size_t)c * V + j] = a[c] * dP;
                    }
                    dg[ix_g(&d, b, t, hv, c)] = gt[c] >= -5.0 ? acc : 0.0;
                }
                for (int j = 0; j < V; ++j) dv[ix_v(&d, b, t, hv, j)] = de[j];
                dbeta[ix_beta(&d, b, t, hv)] = db;
                for (int c = 0; c < K; ++c) {
                    dq_hv[ix_g(&d, b, t, hv, c)] = scale * dqs[c];
                    dk_hv[ix_g(&d, b, t, hv, c)] = dkt[c];
                }
            }
        }
        if (dh0) memcpy(dh0 + ix_state(&d, b, hv), dS, KV * sizeof(double));
        free(ckpt); free(states); free(dS); free(P);
        free(qt); free(kt); free(gt); free(vt); free(e); free(de); free(dot); free(a);
        free(dkt); free(dqs);
    }

    /* sum dq, dk over the value heads of each group (GVA) */
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < T; ++t)
            for (int h = 0; h < H; ++h)
                for (int c = 0; c < K; ++c) {
                    double sq = 0.0, sk = 0.0;
                    for (int i = 0; i < G; ++i) {
                        sq += dq_hv[ix_g(&d, b, t, h * G + i, c)];
                        sk += dk_hv[ix_g(&d, b, t, h * G + i, c)];
                    }
                    dq[ix_qk(&d, b, t, h, c)] = sq;
                    dk[ix_qk(&d, b, t, h, c)] = sk;
                }
    free(dq_hv);
    free(dk_hv);
}

/* ------------------------------------------------------------------------ */
/* Chunk form (K3 row L2).                                                   */
/*                                                                           */
/* Inside a chunk of rows r = 0..n-1 starting from state S:                  */
/*   (1) G_r = sum_{s<=r} max(g_s,-5)                 (per key channel)      */
/*   (2) A[i][j] = beta_i sum_c k_ic k_jc exp(G_ic - G_jc),  j < i           */
/*   (3) T = (I + A)^{-1} (forward substitution);                            */
/*       W = T diag(beta) (k o exp(G)),  U = T diag(beta) v                  */
/*   (4) delta = U - W S                                                     */
/*       Aqk[r][j] = sum_c qs_rc k_jc exp(G_rc - G_jc),  j <= r              */
/*       O = (qs o exp(G)) S + Aqk delta                                     */
/*       S <- diag(exp(G_last)) S + sum_j (k_j o exp(G_last - G_j)) delta_j^T*/
/* ------------------------------------------------------------------------ */

/* The step (1)-(3) quantities of one chunk of n rows.  Inputs are the rows of
 * one head: qs (n x K, already scaled), k (n x K), v (n x V), g (n x K),
 * beta (n).  Outputs (any may be NULL): Gc (n x K), A (n x n), Tm (n x n),
 * W (n x K), U (n x V), Aqk (n x n). */
static void chunk_wy(int n, int K, int V, const double* qs, const double* k,
                     const double* v, const double* g, const double* beta, double* Gc,
                     double* A, double* Tm, double* W, double* U, double* Aqk) {
    for (int c = 0; c < K; ++c) {
        double acc = 0.0;
        for (int r = 0; r < n; ++r) {
            acc += gate_hat(g[(size_t)r * K + c]);
            Gc[(size_t)r * K + c] = acc;
        }
    }
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < n; ++j) {
            double a = 0.0, aq = 0.0;
            if (j <= i) {
                for (int c = 0; c < K; ++c) {
                    double dec = exp(Gc[(size_t)i * K + c] - Gc[(size_t)j * K + c]);
                    a += k[(size_t)i * K + c] * k[(size_t)j * K + c] * dec;
                    aq += qs[(size_t)i * K + c] * k[(size_t)j * K + c] * dec;
                }
            }
            A[(size_t)i * n + j] = j < i ? beta[i] * a : 0.0;
            Aqk[(size_t)i * n + j] = j <= i ? aq : 0.0;
        }
    /* T = (I + A)^{-1}: column j solves (I + A) x = e_j top to bottom */
    for (int j = 0; j < n; ++j)
        for (int i = 0; i < n; ++i) {
            if (i < j) { Tm[(size_t)i * n + j] = 0.0; continue; }
            if (i == j) { Tm[(size_t)i * n + j] = 1.0; continue; }
            double acc = 0.0;
            for (int m = j; m < i; ++m) acc += A[(size_t)i * n + m] * Tm[(size_t)m * n + j];
            Tm[(size_t)i * n + j] = -acc;
        }
    for (int i = 0; i < n; ++i) {
        for (int c = 0; c < K; ++c) {
            double acc = 0.0;
            for (int m = 0; m <= i; ++m)
                acc += Tm[(size_t)i * n + m] * beta[m] * k[(size_t)m * K + c] *
                       exp(Gc[(size_t)m * K + c]);
            W[(size_t)i * K + c] = acc;
        }
        for (int j = 0; j < V; ++j) {
            double acc = 0.0;
            for (int m = 0; m <= i; ++m) acc += Tm[(size_t)i * n + m] * beta[m] * v[(size_t)m * V + j];
            U[(size_t)i * V + j] = acc;
        }
    }
}

void kda_oracle_chunk_wy(int n, int K, int V, const double* qs, const double* k,
                         const double* v, const double* g, const double* beta, double* Gc,
                         double* A, double* Tm, double* W, double* U, double* Aqk) {
    chunk_wy(n, K, V, qs, k, v, g, beta, Gc, A, Tm, W, U, Aqk);
}

void kda_oracle_fwd_chunked(int B, int T, int H, int HV, int K, int V, double scale,
                            int chunk, const double* q, const double* k, const double* v,
                            const double* g, const double* beta, const double* h0, double* o,
                            double* ht) {
    odims d = {B, T, H, HV, K, V, scale};
    int nheads = B * HV;
    int C = chunk;
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < nheads; ++bh) {
        int b = bh / HV, hv = bh % HV;
        int h = hv / (HV / H);
        size_t KV = (size_t)K * V;
        double* S = (double*)calloc(KV, sizeof(double));
        double* qs = malloc((size_t)C * K * sizeof(double));
        double* kc = malloc((size_t)C * K * sizeof(double));
        double* gc = malloc((size_t)C * K * sizeof(double));
        double* vc = malloc((size_t)C * V * sizeof(double));
        double* bc = malloc((size_t)C * sizeof(double));
        double* Gc = malloc((size_t)C * K * sizeof(double));
        double* A = malloc((size_t)C * C * sizeof(double));
        double* Tm = malloc((size_t)C * C * sizeof(double));
        double* W = malloc((size_t)C * K * sizeof(double));
        double* U = malloc((size_t)C * V * sizeof(double));
        double* Aqk = malloc((size_t)C * C * sizeof(double));
        double* delta = malloc((size_t)C * V * sizeof(double));
        if (h0) memcpy(S, h0 + ix_state(&d, b, hv), KV * sizeof(double));
        for (int t0 = 0; t0 < T; t0 += C) {
            int n = T - t0 < C ? T - t0 : C;
            for (int r = 0; r < n; ++r) {
                int t = t0 + r;
                for (int c = 0; c < K; ++c) {
                    qs[(size_t)r * K + c] = scale * q[ix_qk(&d, b, t, h, c)];
                    kc[(size_t)r * K + c] = k[ix_qk(&d, b, t, h, c)];
                    gc[(size_t)r * K + c] = g[ix_g(&d, b, t, hv, c)];
                }
                for (int j = 0; j < V; ++j) vc[(size_t)r * V + j] = v[ix_v(&d, b, t, hv, j)];
                bc[r] = beta[ix_beta(&d, b, t, hv)];
            }
            chunk_wy(n, K, V, qs, kc, vc, gc, bc, Gc, A, Tm, W, U, Aqk);
            /* delta = U - W S */
            for (int r = 0; r < n; ++r)
                for (int j = 0; j < V; ++j) {
                    double acc = 0.0;
                    for (int c = 0; c < K; ++c) acc += W[(size_t)r * K + c] * S[(size_t)c * V + j];
                    delta[(size_t)r * V + j] = U[(size_t)r * V + j] - acc;
                }
            /* O = (qs o exp(G)) S + Aqk delta */
            for (int r = 0; r < n; ++r)
                for (int j = 0; j < V; ++j) {
                    double acc = 0.0;
                    for (int c = 0; c < K; ++c)
                        acc += qs[(size_t)r * K + c] * exp(Gc[(size_t)r * K + c]) * S[(size_t)c * V + j];
                    for (int m = 0; m <= r; ++m) acc += Aqk[(size_t)r * n + m] * delta[(size_t)m * V + j];
                    o[ix_v(&d, b, t0 + r, hv, j)] = acc;
                }
            /* S <- diag(exp(G_last)) S + sum_m (k_m o exp(G_last - G_m)) delta_m^T */
            for (int c = 0; c < K; ++c) {
                double Gl = Gc[(size_t)(n - 1) * K + c];
                double gam = exp(Gl);
                for (int j = 0; j < V; ++j) {
                    double acc = gam * S[(size_t)c * V + j];
                    for (int m = 0; m < n; ++m)
                        acc += kc[(size_t)m * K + c] * exp(Gl - Gc[(size_t)m * K + c]) *
                               delta[(size_t)m * V + j];
                    S[(size_t)c * V + j] = acc;
                }
            }
        }
        if (ht) memcpy(ht + ix_state(&d, b, hv), S, KV * sizeof(double));
        free(S); free(qs); free(kc); free(gc); free(vc); free(bc); free(Gc); free(A);
        free(Tm); free(W); free(U); free(Aqk); free(delta);
    }
}

/* ------------------------------------------------------------------------ */
/* Decode: one token per head, state updated in place (K3 row L6).           */
/* q, k [B,H,K]; v, o [B,HV,V]; g [B,HV,K]; beta [B,HV]; state [B,HV,K,V].   */
/* ------------------------------------------------------------------------ */
void kda_oracle_step(int B, int H, int HV, int K, int V, double scale, const double* q,
                     const double* k, const double* v, const double* g, const double* beta,
                     double* state, double* o) {
    int nheads = B * HV;
    int G = HV / H;
#pragma omp parallel for schedule(dynamic, 4)
    for (int bh = 0; bh < nheads; ++bh) {
        int b = bh / HV, hv = bh % HV, h = hv / G;
        token_step(K, V, scale, q + ((size_t)b * H + h) * K, k + ((size_t)b * H + h) * K,
                   v + (size_t)bh * V, g + (size_t)bh * K, beta[bh],
                   state + (size_t)bh * K * V, o + (size_t)bh * V, NULL);
    }
}

/* ------------------------------------------------------------------------ */
/* L2 normalisation of q and k over K, and its backward (the "q/k L2-norm"   */
/* variant of the K3 README's test-status table, row L3/L4).  The pages give */
/* no formula beyond the name; the plain reading is x / ||x||_2 per token    */
/* and head, with the norm floored at 1e-12 so that a zero row maps to zero. */
/*   y  = x / max(||x||, eps)                                               */
/*   dx = (dy - y <y, dy>) / ||x||       where ||x|| > eps                   */
/*   dx = dy / eps                       where the floor is active           */
/* rows vectors of length K, contiguous.                                     */
/* ------------------------------------------------------------------------ */
void kda_oracle_l2norm(long rows, int K, const double* x, double* y) {
    for (long r = 0; r < rows; ++r) {
        const double* xr = x + (size_t)r * K;
        double ss = 0.0;
        for (int c = 0; c < K; ++c) ss += xr[c] * xr[c];
        double n = sqrt(ss);
        double den = n > 1e-12 ? n : 1e-12;
        for (int c = 0; c < K; ++c) y[(size_t)r * K + c] = xr[c] / den;
    }
}

void kda_oracle_l2norm_bwd(long rows, int K, const double* x, const double* dy, double* dx) {
    for (long r = 0; r < rows; ++r) {
        const double* xr = x + (size_t)r * K;
        const double* dyr = dy + (size_t)r * K;
        double ss = 0.0;
        for (int c = 0; c < K; ++c) ss += xr[c] * xr[c];
        double n = sqrt(ss);
        if (n > 1e-12) {
            double dot = 0.0;
            for (int c = 0; c < K; ++c) dot += (xr[c] / n) * dyr[c];
            for (int c = 0; c < K; ++c) dx[(size_t)r * K + c] = (dyr[c] - (xr[c] / n) * dot) / n;
        } else {
            for (int c = 0; c < K; ++c) dx[(size_t)r * K + c] = dyr[c] / 1e-12;
        }
    }
}
