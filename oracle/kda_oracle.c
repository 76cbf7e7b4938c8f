/*
 * kda_oracle.c -- plain fp64 CPU oracle of the Kimi Delta Attention (KDA)
 * mixer core.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg call it; the CUDA library never does, and the
 * two share no code.
 *
 * Everything is computed token by token in double precision, in the order the
 * sources state it:
 *
 *   "Kimi Delta Attention (KDA) -- analysis & C kernel plan" (sqliteai/waste,
 *   docs/KDA.md), section "The KDA layer, precisely":
 *       q = SiLU(ShortConv_4(q_raw)), same for k and v;
 *       g = fused_kda_gate(...); beta = sigmoid(b);
 *       o, S = KDA_recurrence(q, k, v, g, beta, S)   (q, k L2-normalised inside);
 *       o = RMSNormGated(o, gate)
 *   same page, section "Recurrence":
 *       S' = Diag(exp(g_t)) S_{t-1};  S_t = S' + beta_t k_t (v_t - S'^T k_t)^T;
 *       o_t = S_t^T q_t   (q L2-normalised, then times K^-0.5)
 *   "ferrox-models 0.8.0, module kda" (docs.rs), module overview: L2-normalise
 *   q and k with eps 1e-6, then scale q by head_dim^-0.5; gate per (head,
 *   key-dim); output gate activation is sigmoid; conv is a depthwise causal
 *   Conv1d with padding kernel_size-1 and no bias.
 *   "Kimi K3 - Retention gate - OpenModelAtlas", excerpt of gate.py
 *   (naive_kda_lowerbound_gate): g = lower_bound * sigmoid(exp(A_log) * (z + dt_bias)).
 *   The earlier Kimi-Linear gate (gate_kind 1), "Kimi Delta Attention (KDA) --
 *   analysis & C kernel plan" (status note and "The KDA layer, precisely":
 *   fused_kda_gate(..., A_log, bias=dt_bias)): g = -exp(A_log) * softplus(z + dt_bias).
 *
 * Readings where the sources leave a step open (each also listed in the design
 * notes of the repository):
 *   - L2 norm: x * (sum x^2 + eps)^(-1/2).
 *   - Conv: PyTorch Conv1d cross-correlation with left padding 3; tap 3 weighs
 *     the current token, tap 0 the token three steps back.
 *   - Conv ring: the three last RAW (pre-conv) inputs per plane, slot 0 oldest.
 *   - RMSNormGated: normalise over head_dim, times weight[i], times
 *     sigmoid(gate); one weight vector of length head_dim shared by all heads.
 *   - State S per head is [key][value]; the decay scales key rows.
 *
 * Layouts (all row-major, double):
 *   token tensors q,k,v,z,gout  [T][H*D]   channel c = h*D + i
 *   b                           [T][H]
 *   S                           [n][H][D][D]   S[key][value]
 *   ring                        [n][3 planes q,k,v][3 slots][H*D]
 *   conv_w                      [3 planes][H*D][4 taps]
 *
 * Work is split over independent (sequence, head) units with pthreads; each
 * unit is computed by one thread in a fixed order, so the result does not
 * depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define KDAO_CONV_K 4
#define KDAO_RING 3

typedef struct {
    int32_t num_heads;     /* H */
    int32_t head_dim;      /* D */
    double gate_lower_bound;
    double l2_eps;
    double norm_eps;
    double q_scale;        /* 0 -> D^-1/2 */
    const double* conv_w;  /* [3][H*D][4] */
    const double* A_log;   /* [H] */
    const double* dt_bias; /* [H*D] */
    const double* norm_w;  /* [D] */
    int32_t gate_kind;     /* 0: lower-bounded sigmoid gate; 1: -exp(A_log) softplus(z + dt_bias) */
} kdao_params;

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }
/* log(1 + e^x) without overflow */
static double softplus(double x) { return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x)); }

/* ------------------------------------------------------------------------ */
/* Thread pool helper: run fn(i, ctx) for i in [0, n) over nthreads threads. */
typedef void (*unit_fn)(int64_t unit, void* ctx);
typedef struct {
    unit_fn fn;
    void* ctx;
    int64_t n;
    int64_t next;
    pthread_mutex_t mu;
} pool_t;

static void* pool_worker(void* arg) {
    pool_t* p = (pool_t*)arg;
    for (;;) {
        pthread_mutex_lock(&p->mu);
        int64_t u = p->next++;
        pthread_mutex_unlock(&p->mu);
        if (u >= p->n) break;
        p->fn(u, p->ctx);
    }
    return NULL;
}

static void run_units(int64_t n, int nthreads, unit_fn fn, void* ctx) {
    if (n <= 0) return;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n) nthreads = (int)n;
    pool_t p;
    p.fn = fn; p.ctx = ctx; p.n = n; p.next = 0;
    pthread_mutex_init(&p.mu, NULL);
    if (nthreads == 1) {
        pool_worker(&p);
    } else {
        pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
        for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, pool_worker, &p);
        for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
        free(th);
    }
    pthread_mutex_destroy(&p.mu);
}

/* ------------------------------------------------------------------------ */
/* One recurrence step for one head (Recurrence section of the waste page).
 *   Sp = Diag(exp(g)) S ; u = Sp^T k ; S = Sp + beta k (v - u)^T ; o = S^T q
 * S is D x D, row = key index, column = value index.  u and tmp are scratch. */
static void recurrence_step(int D, double* S, const double* q, const double* k,
                            const double* v, const double* g, double beta,
                            double* o, double* u) {
    for (int i = 0; i < D; ++i) {          /* S' = Diag(exp(g)) S */
        double e = exp(g[i]);
        for (int j = 0; j < D; ++j) S[i * D + j] *= e;
    }
    for (int j = 0; j < D; ++j) u[j] = 0.0; /* u = S'^T k */
    for (int i = 0; i < D; ++i)
        for (int j = 0; j < D; ++j) u[j] += S[i * D + j] * k[i];
    for (int i = 0; i < D; ++i)             /* S = S' + beta k (v - u)^T */
        for (int j = 0; j < D; ++j) S[i * D + j] += beta * k[i] * (v[j] - u[j]);
    for (int j = 0; j < D; ++j) o[j] = 0.0; /* o = S^T q */
    for (int i = 0; i < D; ++i)
        for (int j = 0; j < D; ++j) o[j] += S[i * D + j] * q[i];
}

/* ------------------------------------------------------------------------ */
/* Core recurrence on already transformed inputs.
 * q,k,v,g [T][H][D] ; beta [T][H] ; S0 [H][D][D] or NULL (zero) ; S out
 * [H][D][D] ; o out [T][H][D].  One unit per head. */
typedef struct {
    int T, H, D;
    const double *q, *k, *v, *g, *beta, *S0;
    double *S, *o;
} core_ctx;

static void core_unit(int64_t h, void* vctx) {
    core_ctx* c = (core_ctx*)vctx;
    int D = c->D, H = c->H;
    double* S = c->S + (size_t)h * D * D;
    if (c->S0) memcpy(S, c->S0 + (size_t)h * D * D, sizeof(double) * D * D);
    else memset(S, 0, sizeof(double) * D * D);
    double* u = (double*)malloc(sizeof(double) * D);
    for (int t = 0; t < c->T; ++t) {
        size_t off = ((size_t)t * H + h) * D;
        recurrence_step(D, S, c->q + off, c->k + off, c->v + off, c->g + off,
                        c->beta[(size_t)t * H + h], c->o + off, u);
    }
    free(u);
}

int kdao_core(int T, int H, int D, const double* q, const double* k, const double* v,
              const double* g, const double* beta, const double* S0, double* S, double* o,
              int nthreads) {
    if (T < 0 || H <= 0 || D <= 0) return 1;
    core_ctx c = {T, H, D, q, k, v, g, beta, S0, S, o};
    run_units(H, nthreads, core_unit, &c);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Chunked form of the same recurrence (the "chunked UT transform" with a
 * per-channel cumulative log gate Gcum, described on the memra-engine page,
 * section PREFILL DISPATCH, and on the retention-gate page, section "Why").
 * It is an independent route to the same numbers and exists to pin the
 * algebra the tensor-core kernel relies on.  Per chunk of Lc <= C tokens,
 * with G_r = sum_{s<=r} g_s inside the chunk (per key channel):
 *   pair (r, s), s <= r, s in sub-tile b, ref = last token of sub-tile b:
 *     A[r][s] = beta_r * sum_i k_ri e^{G_ri - G_ref,i} * k_si e^{G_ref,i - G_si}   (s < r)
 *     P[r][s] =          sum_i q_ri e^{G_ri - G_ref,i} * k_si e^{G_ref,i - G_si}   (s <= r)
 *   T = (I + A)^{-1} Diag(beta)        (forward substitution)
 *   W = T (k * e^{G}) ;  U0 = T v ;  U = U0 - W S0
 *   O = (q * e^{G}) S0 + P U
 *   S_C = Diag(e^{G_last}) S0 + (k * e^{G_last - G})^T U
 * All exponents above are <= 0 except inside a diagonal sub-tile. */
typedef struct {
    int T, H, D, C, ST;
    const double *q, *k, *v, *g, *beta, *S0;
    double *S, *o;
} chunk_ctx;

static void chunk_unit(int64_t h, void* vctx) {
    chunk_ctx* c = (chunk_ctx*)vctx;
    const int D = c->D, H = c->H, C = c->C, ST = c->ST;
    double* S = c->S + (size_t)h * D * D;
    if (c->S0) memcpy(S, c->S0 + (size_t)h * D * D, sizeof(double) * D * D);
    else memset(S, 0, sizeof(double) * D * D);
    double* G = (double*)malloc(sizeof(double) * C * D);
    double* A = (double*)malloc(sizeof(double) * C * C);
    double* P = (double*)malloc(sizeof(double) * C * C);
    double* Tm = (double*)malloc(sizeof(double) * C * C);
    double* Wm = (double*)malloc(sizeof(double) * C * D);
    double* U = (double*)malloc(sizeof(double) * C * D);
    double* Snew = (double*)malloc(sizeof(double) * D * D);
#define IDX(t, i) (((size_t)(t) * H + h) * D + (i))
    for (int t0 = 0; t0 < c->T; t0 += C) {
        int Lc = c->T - t0 < C ? c->T - t0 : C;
        for (int i = 0; i < D; ++i) {
            double acc = 0.0;
            for (int r = 0; r < Lc; ++r) { acc += c->g[IDX(t0 + r, i)]; G[r * D + i] = acc; }
        }
        for (int r = 0; r < Lc; ++r) {
            for (int s = 0; s <= r; ++s) {
                int b = s / ST;
                int ref = b * ST + ST - 1;
                if (ref > Lc - 1) ref = Lc - 1;
                double a = 0.0, pq = 0.0;
                for (int i = 0; i < D; ++i) {
                    double right = c->k[IDX(t0 + s, i)] * exp(G[ref * D + i] - G[s * D + i]);
                    double lscale = exp(G[r * D + i] - G[ref * D + i]);
                    a += c->k[IDX(t0 + r, i)] * lscale * right;
                    pq += c->q[IDX(t0 + r, i)] * lscale * right;
                }
                A[r * C + s] = (s < r) ? c->beta[(size_t)(t0 + r) * H + h] * a : 0.0;
                P[r * C + s] = pq;
            }
            for (int s = r + 1; s < Lc; ++s) { A[r * C + s] = 0.0; P[r * C + s] = 0.0; }
        }
        /* (I + A) T = Diag(beta): row r of T = beta_r e_r - sum_{s<r} A[r][s] T_s */
        for (int r = 0; r < Lc; ++r) {
            for (int j = 0; j < Lc; ++j)
                Tm[r * C + j] = (j == r) ? c->beta[(size_t)(t0 + r) * H + h] : 0.0;
            for (int s = 0; s < r; ++s) {
                double ars = A[r * C + s];
                for (int j = 0; j < Lc; ++j) Tm[r * C + j] -= ars * Tm[s * C + j];
            }
        }
        /* W = T (k e^G), U = T v - W S0 */
        for (int r = 0; r < Lc; ++r) {
            for (int i = 0; i < D; ++i) {
                double w = 0.0, u0 = 0.0;
                for (int s = 0; s < Lc; ++s) {
                    w += Tm[r * C + s] * c->k[IDX(t0 + s, i)] * exp(G[s * D + i]);
                    u0 += Tm[r * C + s] * c->v[IDX(t0 + s, i)];
                }
                Wm[r * D + i] = w;
                U[r * D + i] = u0;
            }
        }
        for (int r = 0; r < Lc; ++r)
            for (int j = 0; j < D; ++j) {
                double ws = 0.0;
                for (int i = 0; i < D; ++i) ws += Wm[r * D + i] * S[i * D + j];
                U[r * D + j] -= ws;
            }
        /* O = (q e^G) S0 + P U */
        for (int r = 0; r < Lc; ++r)
            for (int j = 0; j < D; ++j) {
                double acc = 0.0;
                for (int i = 0; i < D; ++i) acc += c->q[IDX(t0 + r, i)] * exp(G[r * D + i]) * S[i * D + j];
                for (int s = 0; s <= r; ++s) acc += P[r * C + s] * U[s * D + j];
                c->o[IDX(t0 + r, j)] = acc;
            }
        /* S_C = Diag(e^{G_last}) S0 + (k e^{G_last - G})^T U */
        for (int i = 0; i < D; ++i) {
            double glast = G[(Lc - 1) * D + i];
            for (int j = 0; j < D; ++j) {
                double acc = exp(glast) * S[i * D + j];
                for (int s = 0; s < Lc; ++s)
                    acc += c->k[IDX(t0 + s, i)] * exp(glast - G[s * D + i]) * U[s * D + j];
                Snew[i * D + j] = acc;
            }
        }
        memcpy(S, Snew, sizeof(double) * D * D);
    }
#undef IDX
    free(G); free(A); free(P); free(Tm); free(Wm); free(U); free(Snew);
}

int kdao_chunked_core(int T, int H, int D, int C, int subtile, const double* q, const double* k,
                      const double* v, const double* g, const double* beta, const double* S0,
                      double* S, double* o, int nthreads) {
    if (T < 0 || H <= 0 || D <= 0 || C <= 0 || subtile <= 0) return 1;
    chunk_ctx c = {T, H, D, C, subtile < C ? subtile : C, q, k, v, g, beta, S0, S, o};
    run_units(H, nthreads, chunk_unit, &c);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Pre-stage for one token of one head: conv + SiLU on the three planes,
 * L2 normalisation of q and k, q scaling, gate and beta.
 * xwin[p][j] is the raw input of plane p at relative step j (j = 3 current).
 * Outputs qh, kh, vh, g [D] and *beta. */
static void prestage_token(const kdao_params* p, int h, const double* xwin /*[3][4][D]*/,
                           const double* zrow, double braw,
                           double* qh, double* kh, double* vh, double* g, double* beta) {
    const int D = p->head_dim, W = p->num_heads * p->head_dim;
    double* outs[3] = {qh, kh, vh};
    for (int pl = 0; pl < 3; ++pl) {
        for (int i = 0; i < D; ++i) {
            int ch = h * D + i;
            const double* w = p->conv_w + ((size_t)pl * W + ch) * KDAO_CONV_K;
            double acc = 0.0;
            for (int j = 0; j < KDAO_CONV_K; ++j) acc += w[j] * xwin[((size_t)pl * KDAO_CONV_K + j) * D + i];
            outs[pl][i] = acc * sigmoid(acc); /* SiLU */
        }
    }
    double sq = 0.0, sk = 0.0;
    for (int i = 0; i < D; ++i) { sq += qh[i] * qh[i]; sk += kh[i] * kh[i]; }
    double scale = p->q_scale != 0.0 ? p->q_scale : 1.0 / sqrt((double)D);
    double rq = 1.0 / sqrt(sq + p->l2_eps), rk = 1.0 / sqrt(sk + p->l2_eps);
    for (int i = 0; i < D; ++i) { qh[i] = qh[i] * rq * scale; kh[i] = kh[i] * rk; }
    double ea = exp(p->A_log[h]);
    for (int i = 0; i < D; ++i) {
        int ch = h * D + i;
        if (p->gate_kind == 1) /* Kimi-Linear decay gate, unbounded below */
            g[i] = -ea * softplus(zrow[i] + p->dt_bias[ch]);
        else
            g[i] = p->gate_lower_bound * sigmoid(ea * (zrow[i] + p->dt_bias[ch]));
    }
    *beta = sigmoid(braw);
}

/* RMSNormGated for one (token, head): o = x / sqrt(mean(x^2) + eps) * w * sigmoid(gate) */
static void rmsnorm_gated_head(int D, double eps, const double* x, const double* gate,
                               const double* w, double* o) {
    double ss = 0.0;
    for (int i = 0; i < D; ++i) ss += x[i] * x[i];
    double r = 1.0 / sqrt(ss / D + eps);
    for (int i = 0; i < D; ++i) o[i] = x[i] * r * w[i] * sigmoid(gate[i]);
}

/* ------------------------------------------------------------------------ */
/* Full mixer.  Units are (sequence, head).  Optional intermediate outputs
 * (any may be NULL): qh,kh,vh,g,o_core [T][H*D], beta [T][H]. */
typedef struct {
    const kdao_params* p;
    int n_seqs;
    const int64_t* cu;
    const double *q, *k, *v, *z, *b, *gout, *S_in, *ring_in;
    double *S_out, *ring_out, *o, *qh_out, *kh_out, *vh_out, *g_out, *beta_out, *ocore_out;
} mixer_ctx;

static void mixer_unit(int64_t unit, void* vctx) {
    mixer_ctx* c = (mixer_ctx*)vctx;
    const kdao_params* p = c->p;
    const int H = p->num_heads, D = p->head_dim, W = H * D;
    int n = (int)(unit / H), h = (int)(unit % H);
    int64_t bos = c->cu[n], eos = c->cu[n + 1], L = eos - bos;
    const double* xs[3] = {c->q, c->k, c->v};

    double* S = (double*)malloc(sizeof(double) * D * D);
    const size_t soff = ((size_t)n * H + h) * D * D;
    if (c->S_in) memcpy(S, c->S_in + soff, sizeof(double) * D * D);
    else memset(S, 0, sizeof(double) * D * D);

    double* xwin = (double*)malloc(sizeof(double) * 3 * KDAO_CONV_K * D);
    double *qh = (double*)malloc(sizeof(double) * D), *kh = (double*)malloc(sizeof(double) * D);
    double *vh = (double*)malloc(sizeof(double) * D), *g = (double*)malloc(sizeof(double) * D);
    double *oc = (double*)malloc(sizeof(double) * D), *u = (double*)malloc(sizeof(double) * D);
    double *orow = (double*)malloc(sizeof(double) * D);

    for (int64_t tau = 0; tau < L; ++tau) {
        int64_t t = bos + tau;
        /* causal window: relative step j in [0,4) reads local index tau-3+j */
        for (int pl = 0; pl < 3; ++pl)
            for (int j = 0; j < KDAO_CONV_K; ++j) {
                int64_t src = tau - (KDAO_CONV_K - 1) + j;
                for (int i = 0; i < D; ++i) {
                    int ch = h * D + i;
                    double x;
                    if (src >= 0) x = xs[pl][(size_t)(bos + src) * W + ch];
                    else if (c->ring_in)
                        x = c->ring_in[(((size_t)n * 3 + pl) * KDAO_RING + (size_t)(KDAO_RING + src)) * W + ch];
                    else x = 0.0;
                    xwin[((size_t)pl * KDAO_CONV_K + j) * D + i] = x;
                }
            }
        double beta;
        prestage_token(p, h, xwin, c->z + (size_t)t * W + (size_t)h * D,
                       c->b[(size_t)t * H + h], qh, kh, vh, g, &beta);
        recurrence_step(D, S, qh, kh, vh, g, beta, oc, u);
        rmsnorm_gated_head(D, p->norm_eps, oc, c->gout + (size_t)t * W + (size_t)h * D, p->norm_w, orow);
        size_t ro = (size_t)t * W + (size_t)h * D;
        memcpy(c->o + ro, orow, sizeof(double) * D);
        if (c->qh_out) memcpy(c->qh_out + ro, qh, sizeof(double) * D);
        if (c->kh_out) memcpy(c->kh_out + ro, kh, sizeof(double) * D);
        if (c->vh_out) memcpy(c->vh_out + ro, vh, sizeof(double) * D);
        if (c->g_out) memcpy(c->g_out + ro, g, sizeof(double) * D);
        if (c->ocore_out) memcpy(c->ocore_out + ro, oc, sizeof(double) * D);
        if (c->beta_out) c->beta_out[(size_t)t * H + h] = beta;
    }
    memcpy(c->S_out + soff, S, sizeof(double) * D * D);

    /* final ring: the last three raw inputs of the sequence; when the
     * sequence is shorter than three, the older slots come from ring_in */
    if (c->ring_out) {
        for (int pl = 0; pl < 3; ++pl)
            for (int s = 0; s < KDAO_RING; ++s) {
                int64_t src = L - KDAO_RING + s;
                for (int i = 0; i < D; ++i) {
                    int ch = h * D + i;
                    double x;
                    if (src >= 0) x = xs[pl][(size_t)(bos + src) * W + ch];
                    else if (c->ring_in)
                        x = c->ring_in[(((size_t)n * 3 + pl) * KDAO_RING + (size_t)(KDAO_RING + src)) * W + ch];
                    else x = 0.0;
                    c->ring_out[(((size_t)n * 3 + pl) * KDAO_RING + s) * W + ch] = x;
                }
            }
    }
    free(S); free(xwin); free(qh); free(kh); free(vh); free(g); free(oc); free(u); free(orow);
}

int kdao_mixer(const kdao_params* p, int n_seqs, const int64_t* cu_seqlens,
               const double* q, const double* k, const double* v, const double* z,
               const double* b, const double* gout, const double* S_in, double* S_out,
               const double* ring_in, double* ring_out, double* o,
               double* qh_out, double* kh_out, double* vh_out, double* g_out,
               double* beta_out, double* ocore_out, int nthreads) {
    if (!p || p->num_heads <= 0 || p->head_dim <= 0 || n_seqs < 0 || !cu_seqlens) return 1;
    if (cu_seqlens[0] != 0) return 1;
    for (int n = 0; n < n_seqs; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return 1;
    /* ring_out may alias ring_in: take a private copy of ring_in first */
    double* ring_copy = NULL;
    const double* rin = ring_in;
    if (ring_in && ring_out == ring_in) {
        size_t nr = (size_t)n_seqs * 3 * KDAO_RING * p->num_heads * p->head_dim;
        ring_copy = (double*)malloc(sizeof(double) * (nr ? nr : 1));
        memcpy(ring_copy, ring_in, sizeof(double) * nr);
        rin = ring_copy;
    }
    mixer_ctx c = {p, n_seqs, cu_seqlens, q, k, v, z, b, gout, S_in, rin,
                   S_out, ring_out, o, qh_out, kh_out, vh_out, g_out, beta_out, ocore_out};
    run_units((int64_t)n_seqs * p->num_heads, nthreads, mixer_unit, &c);
    free(ring_copy);
    return 0;
}

/* Stand-alone RMSNormGated over [rows][H*D] (used to pin the epilogue). */
int kdao_rmsnorm_gated(int64_t rows, int H, int D, double eps, const double* x,
                       const double* gate, const double* w, double* o) {
    for (int64_t r = 0; r < rows; ++r)
        for (int h = 0; h < H; ++h) {
            size_t off = (size_t)r * H * D + (size_t)h * D;
            rmsnorm_gated_head(D, eps, x + off, gate + off, w, o + off);
        }
    return 0;
}
