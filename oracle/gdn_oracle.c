/*
 * gdn_oracle.c -- plain fp64 CPU oracle for the gated delta-rule (GDN) recurrence.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark load this library. The CUDA library never links, includes or calls
 * anything here, and this file includes nothing from it.
 *
 * Sources (AWS Neuron NKI library API pages):
 *   "GDN CTE Kernel API Reference"  -- chunked prefill: inputs q,k [B,Hk,S,Dk],
 *       v [B,Hv,S,Dv], g_log and beta [B,Hv,S], scale, optional fp32 recurrent state
 *       [B,Hv,Dk,Dv]; value head h reads key/query head h // (Hv/Hk) (Notes).
 *   "GDN TKG Kernel API Reference"  -- fused decode step: l2norm(q,k),
 *       beta = sigmoid(b), g = -exp(A_log) * softplus(a + dt_bias), RMSNormGated(out, z),
 *       exp(g) and the 1/sqrt(K) q-scale applied inside (Background, Notes, Dimensions).
 *
 * The pages print no formula. The recurrence used here is the gated delta rule with a
 * state S laid out [Dk, Dv]:
 *     S_t = exp(g_t) (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,
 *     o_t = scale * S_t^T q_t        (the output reads the updated state).
 *
 * Functions and what pins them (tests/test_oracle_pins.py):
 *   gdn_oracle_prefill             -- the recurrence written out token by token.
 *       Pinned by dense brute-force products, closed forms (identity, pure decay,
 *       exact write/read, orthonormal memory, first token, reset), a hand-worked
 *       example in tests/golden/ and structural invariants (GQA map, head
 *       independence, split-and-carry).
 *   gdn_oracle_prefill_chunked     -- the chunk-parallel (WY) form, derived algebra;
 *       pinned against the recurrence for chunk sizes 1..128 and ragged tails.
 *   gdn_oracle_unit_lower_inverse  -- (I + A)^-1 by forward substitution; pinned by
 *       T(I + A) = I and the finite Neumann series of the nilpotent A.
 *   gdn_oracle_decode_step         -- the fused decode step. Its recurrence core is
 *       pinned against the prefill recurrence and a hand-worked example; the gates by
 *       closed forms. The RMSNormGated epilogue's eps and its norm-then-gate order
 *       are not stated on the pages: for those two choices, parity unpinned
 *       (closed forms pin the formula as read, not the reading itself).
 *   gdn_oracle_conv1d_decode       -- the depthwise causal conv1d decode token
 *       ("GDN Block TKG Kernel API Reference"); pinned by impulse responses, the
 *       shift register and pass-through cases. Its window order and the absence of a
 *       bias are readings (the page gives shapes only).
 *
 * Everything is fp64. Inputs arrive as double (bf16/fp32 -> double is exact).
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Work split over independent (batch, value-head) units.                     */
/* ------------------------------------------------------------------------ */

typedef void (*unit_fn)(void* ctx, long unit);

typedef struct {
    unit_fn fn;
    void* ctx;
    long first, last; /* [first, last) */
} span_t;

static void* run_span(void* p) {
    span_t* s = (span_t*)p;
    for (long u = s->first; u < s->last; ++u) s->fn(s->ctx, u);
    return NULL;
}

static void for_each_unit(unit_fn fn, void* ctx, long n_units, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n_units) nthreads = (int)(n_units > 0 ? n_units : 1);
    if (nthreads == 1) {
        for (long u = 0; u < n_units; ++u) fn(ctx, u);
        return;
    }
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    span_t* sp = (span_t*)malloc(sizeof(span_t) * (size_t)nthreads);
    long per = n_units / nthreads, extra = n_units % nthreads, at = 0;
    for (int i = 0; i < nthreads; ++i) {
        long n = per + (i < extra ? 1 : 0);
        sp[i].fn = fn; sp[i].ctx = ctx; sp[i].first = at; sp[i].last = at + n;
        at += n;
        pthread_create(&th[i], NULL, run_span, &sp[i]);
    }
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    free(th);
    free(sp);
}

/* ------------------------------------------------------------------------ */
/* Prefill, token by token (the definition).                                 */
/* ------------------------------------------------------------------------ */

typedef struct {
    const double *q, *k, *v, *g_log, *beta, *state0;
    double scale;
    int B, Hk, Hv, S, Dk, Dv, C;
    double *out, *state;
} prefill_ctx;

/* One (b, h) unit. q,k row t of head kh = h / (Hv/Hk) ("GDN CTE Kernel API
 * Reference", Notes: value head h reads key/query head h // (Hv//Hk)). */
static void prefill_unit(void* vctx, long unit) {
    prefill_ctx* c = (prefill_ctx*)vctx;
    const int b = (int)(unit / c->Hv), h = (int)(unit % c->Hv);
    const int kh = h / (c->Hv / c->Hk);
    const int S = c->S, Dk = c->Dk, Dv = c->Dv;
    const double* q = c->q + ((size_t)b * c->Hk + kh) * (size_t)S * Dk;
    const double* k = c->k + ((size_t)b * c->Hk + kh) * (size_t)S * Dk;
    const double* v = c->v + ((size_t)b * c->Hv + h) * (size_t)S * Dv;
    const double* g = c->g_log + ((size_t)b * c->Hv + h) * (size_t)S;
    const double* be = c->beta + ((size_t)b * c->Hv + h) * (size_t)S;
    double* out = c->out + ((size_t)b * c->Hv + h) * (size_t)S * Dv;
    double* St = c->state + ((size_t)b * c->Hv + h) * (size_t)Dk * Dv; /* [Dk][Dv] */

    /* Initial state: the supplied one, else zero ("GDN CTE Kernel API Reference",
     * :param recurrent_state:). */
    if (c->state0) memcpy(St, c->state0 + ((size_t)b * c->Hv + h) * (size_t)Dk * Dv,
                          sizeof(double) * (size_t)Dk * Dv);
    else memset(St, 0, sizeof(double) * (size_t)Dk * Dv);

    double* x = (double*)malloc(sizeof(double) * (size_t)Dv);
    for (int t = 0; t < S; ++t) {
        const double* kt = k + (size_t)t * Dk;
        const double* qt = q + (size_t)t * Dk;
        const double* vt = v + (size_t)t * Dv;
        const double alpha = exp(g[t]), bt = be[t];
        /* x = k_t^T S_{t-1}: the row vector that (I - beta k k^T) S needs. */
        for (int j = 0; j < Dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < Dk; ++i) acc += kt[i] * St[(size_t)i * Dv + j];
            x[j] = acc;
        }
        /* S_t = alpha (S_{t-1} - beta k_t x) + beta k_t v_t^T, element by element. */
        for (int i = 0; i < Dk; ++i)
            for (int j = 0; j < Dv; ++j) {
                double* s = &St[(size_t)i * Dv + j];
                *s = alpha * (*s - bt * kt[i] * x[j]) + bt * kt[i] * vt[j];
            }
        /* o_t = scale * S_t^T q_t. */
        for (int j = 0; j < Dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < Dk; ++i) acc += qt[i] * St[(size_t)i * Dv + j];
            out[(size_t)t * Dv + j] = c->scale * acc;
        }
    }
    free(x);
}

/* Returns 0 on success, -1 on bad shapes. */
int gdn_oracle_prefill(const double* q, const double* k, const double* v,
                       const double* g_log, const double* beta, double scale,
                       int B, int Hk, int Hv, int S, int Dk, int Dv,
                       const double* state0, double* out, double* state, int nthreads) {
    if (B < 0 || Hk <= 0 || Hv <= 0 || S < 0 || Dk <= 0 || Dv <= 0 || Hv % Hk != 0) return -1;
    prefill_ctx c = {q, k, v, g_log, beta, state0, scale, B, Hk, Hv, S, Dk, Dv, 0, out, state};
    for_each_unit(prefill_unit, &c, (long)B * Hv, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* (I + A)^-1 for strictly lower-triangular A, by forward substitution.       */
/* ------------------------------------------------------------------------ */

/* A, T: n x n row-major. Solves (I + A) T = I column by column: for column j,
 * T[r,j] = delta_rj - sum_{m<r} A[r,m] T[m,j], rows taken in increasing r. */
void gdn_oracle_unit_lower_inverse(const double* A, int n, double* T) {
    for (int j = 0; j < n; ++j)
        for (int r = 0; r < n; ++r) {
            double acc = (r == j) ? 1.0 : 0.0;
            for (int m = 0; m < r; ++m) acc -= A[(size_t)r * n + m] * T[(size_t)m * n + j];
            T[(size_t)r * n + j] = acc;
        }
}

/* ------------------------------------------------------------------------ */
/* Prefill in chunk-parallel (WY) form -- derived algebra.                    */
/* ------------------------------------------------------------------------ */
/*
 * "GDN CTE Kernel API Reference" computes the recurrence "in chunk-parallel form"
 * with an intra-chunk "(I+A) inverse". The page prints no algebra; this is the
 * derivation from the recurrence above. Writing the token step as
 *     S_t = alpha_t S_{t-1} + k_t u_t^T,   u_t = beta_t (v_t - alpha_t S_{t-1}^T k_t),
 * and, inside a chunk of L tokens with local index r, gamma_r = sum_{i<=r} g_i,
 * Gamma_r = exp(gamma_r), D[r,j] = exp(gamma_r - gamma_j):
 *     A[r,j] = beta_r (k_r . k_j) D[r,j]      (j < r; zero otherwise)
 *     T      = (I + A)^-1
 *     W      = T diag(beta Gamma) K,  U~ = T diag(beta) V,  U = U~ - W S0
 *     P[r,j] = (q_r . k_j) D[r,j]             (j <= r; zero otherwise)
 *     O      = scale (diag(Gamma) Q S0 + P U)
 *     S1     = Gamma_{L-1} S0 + sum_j exp(gamma_{L-1} - gamma_j) k_j u_j^T
 * The last chunk may be shorter than C.
 */
static void chunked_unit(void* vctx, long unit) {
    prefill_ctx* c = (prefill_ctx*)vctx;
    const int b = (int)(unit / c->Hv), h = (int)(unit % c->Hv);
    const int kh = h / (c->Hv / c->Hk);
    const int S = c->S, Dk = c->Dk, Dv = c->Dv, C = c->C;
    const double* q = c->q + ((size_t)b * c->Hk + kh) * (size_t)S * Dk;
    const double* k = c->k + ((size_t)b * c->Hk + kh) * (size_t)S * Dk;
    const double* v = c->v + ((size_t)b * c->Hv + h) * (size_t)S * Dv;
    const double* g = c->g_log + ((size_t)b * c->Hv + h) * (size_t)S;
    const double* be = c->beta + ((size_t)b * c->Hv + h) * (size_t)S;
    double* out = c->out + ((size_t)b * c->Hv + h) * (size_t)S * Dv;
    double* St = c->state + ((size_t)b * c->Hv + h) * (size_t)Dk * Dv;

    if (c->state0) memcpy(St, c->state0 + ((size_t)b * c->Hv + h) * (size_t)Dk * Dv,
                          sizeof(double) * (size_t)Dk * Dv);
    else memset(St, 0, sizeof(double) * (size_t)Dk * Dv);

    double* gam = (double*)malloc(sizeof(double) * (size_t)C);
    double* A = (double*)calloc((size_t)C * C, sizeof(double));
    double* T = (double*)malloc(sizeof(double) * (size_t)C * C);
    double* P = (double*)calloc((size_t)C * C, sizeof(double));
    double* W = (double*)malloc(sizeof(double) * (size_t)C * Dk);
    double* U = (double*)malloc(sizeof(double) * (size_t)C * Dv);
    double* S1 = (double*)malloc(sizeof(double) * (size_t)Dk * Dv);

    for (int c0 = 0; c0 < S; c0 += C) {
        const int L = (S - c0 < C) ? (S - c0) : C;
        const double* Kc = k + (size_t)c0 * Dk;
        const double* Qc = q + (size_t)c0 * Dk;
        const double* Vc = v + (size_t)c0 * Dv;
        const double* gc = g + c0;
        const double* bc = be + c0;
        /* decay cumsum */
        double run = 0.0;
        for (int r = 0; r < L; ++r) { run += gc[r]; gam[r] = run; }
        /* A (strictly lower) and P (lower incl. diagonal) */
        for (int r = 0; r < L; ++r)
            for (int j = 0; j < L; ++j) {
                double kk = 0.0, qk = 0.0;
                for (int i = 0; i < Dk; ++i) {
                    kk += Kc[(size_t)r * Dk + i] * Kc[(size_t)j * Dk + i];
                    qk += Qc[(size_t)r * Dk + i] * Kc[(size_t)j * Dk + i];
                }
                const double d = exp(gam[r] - gam[j]);
                A[(size_t)r * L + j] = (j < r) ? bc[r] * kk * d : 0.0;
                P[(size_t)r * L + j] = (j <= r) ? qk * d : 0.0;
            }
        gdn_oracle_unit_lower_inverse(A, L, T);
        /* W = T diag(beta Gamma) K ; U = T diag(beta) V - W S0 */
        for (int r = 0; r < L; ++r) {
            for (int i = 0; i < Dk; ++i) {
                double acc = 0.0;
                for (int j = 0; j <= r; ++j)
                    acc += T[(size_t)r * L + j] * bc[j] * exp(gam[j]) * Kc[(size_t)j * Dk + i];
                W[(size_t)r * Dk + i] = acc;
            }
            for (int n = 0; n < Dv; ++n) {
                double acc = 0.0;
                for (int j = 0; j <= r; ++j)
                    acc += T[(size_t)r * L + j] * bc[j] * Vc[(size_t)j * Dv + n];
                double ws = 0.0;
                for (int i = 0; i < Dk; ++i) ws += W[(size_t)r * Dk + i] * St[(size_t)i * Dv + n];
                U[(size_t)r * Dv + n] = acc - ws;
            }
        }
        /* O = scale (diag(Gamma) Q S0 + P U) */
        for (int r = 0; r < L; ++r)
            for (int n = 0; n < Dv; ++n) {
                double qs = 0.0, pu = 0.0;
                for (int i = 0; i < Dk; ++i) qs += Qc[(size_t)r * Dk + i] * St[(size_t)i * Dv + n];
                for (int j = 0; j <= r; ++j) pu += P[(size_t)r * L + j] * U[(size_t)j * Dv + n];
                out[(size_t)(c0 + r) * Dv + n] = c->scale * (exp(gam[r]) * qs + pu);
            }
        /* S1 = Gamma_last S0 + sum_j exp(gamma_last - gamma_j) k_j u_j^T */
        const double gl = gam[L - 1];
        for (int i = 0; i < Dk; ++i)
            for (int n = 0; n < Dv; ++n) {
                double acc = exp(gl) * St[(size_t)i * Dv + n];
                for (int j = 0; j < L; ++j)
                    acc += exp(gl - gam[j]) * Kc[(size_t)j * Dk + i] * U[(size_t)j * Dv + n];
                S1[(size_t)i * Dv + n] = acc;
            }
        memcpy(St, S1, sizeof(double) * (size_t)Dk * Dv);
    }
    free(gam); free(A); free(T); free(P); free(W); free(U); free(S1);
}

int gdn_oracle_prefill_chunked(const double* q, const double* k, const double* v,
                               const double* g_log, const double* beta, double scale,
                               int B, int Hk, int Hv, int S, int Dk, int Dv, int C,
                               const double* state0, double* out, double* state, int nthreads) {
    if (B < 0 || Hk <= 0 || Hv <= 0 || S < 0 || Dk <= 0 || Dv <= 0 || C <= 0 || Hv % Hk != 0)
        return -1;
    prefill_ctx c = {q, k, v, g_log, beta, state0, scale, B, Hk, Hv, S, Dk, Dv, C, out, state};
    for_each_unit(chunked_unit, &c, (long)B * Hv, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Fused decode step ("GDN TKG Kernel API Reference").                        */
/* ------------------------------------------------------------------------ */

typedef struct {
    const double *q, *k, *v, *b, *a, *A_log, *dt_bias, *z, *norm_weight, *state_in;
    int BH, H, K, V;
    double eps_l2, eps_rms;
    double *out, *state_out;
} decode_ctx;

/* softplus(x) = log(1 + e^x), in the overflow-free form max(x,0) + log1p(e^-|x|). */
static double softplus(double x) { return (x > 0 ? x : 0.0) + log1p(exp(-fabs(x))); }
static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

static void decode_unit(void* vctx, long bh) {
    decode_ctx* c = (decode_ctx*)vctx;
    const int K = c->K, V = c->V;
    /* BH flattens (batch, v-head) with heads cycling fastest: h = bh mod num_v_heads
     * (Dimensions). */
    const int h = (int)(bh % c->H);
    const double* qr = c->q + (size_t)bh * K;
    const double* kr = c->k + (size_t)bh * K;
    const double* vr = c->v + (size_t)bh * V;
    const double* zr = c->z + (size_t)bh * V;
    const double* S0 = c->state_in + (size_t)bh * K * V;
    double* S1 = c->state_out + (size_t)bh * K * V;
    double* y = c->out + (size_t)bh * V;

    double* qn = (double*)malloc(sizeof(double) * (size_t)K);
    double* kn = (double*)malloc(sizeof(double) * (size_t)K);
    double* x = (double*)malloc(sizeof(double) * (size_t)V);
    double* o = (double*)malloc(sizeof(double) * (size_t)V);

    /* l2norm(q), l2norm(k): x / sqrt(sum x^2 + eps_l2) */
    double sq = 0.0, sk = 0.0;
    for (int i = 0; i < K; ++i) { sq += qr[i] * qr[i]; sk += kr[i] * kr[i]; }
    const double rq = 1.0 / sqrt(sq + c->eps_l2), rk = 1.0 / sqrt(sk + c->eps_l2);
    for (int i = 0; i < K; ++i) { qn[i] = qr[i] * rq; kn[i] = kr[i] * rk; }
    /* beta = sigmoid(b); g = -exp(A_log) * softplus(a + dt_bias); alpha = exp(g) */
    const double beta = sigmoid(c->b[bh]);
    const double g = -exp(c->A_log[h]) * softplus(c->a[bh] + c->dt_bias[h]);
    const double alpha = exp(g);
    /* q-scale 1/sqrt(K), applied here (Notes: not pre-applied upstream) */
    const double scale = 1.0 / sqrt((double)K);

    /* one token of the recurrence: S1 = alpha (S0 - beta k x) + beta k v^T, x = k^T S0 */
    for (int j = 0; j < V; ++j) {
        double acc = 0.0;
        for (int i = 0; i < K; ++i) acc += kn[i] * S0[(size_t)i * V + j];
        x[j] = acc;
    }
    for (int i = 0; i < K; ++i)
        for (int j = 0; j < V; ++j)
            S1[(size_t)i * V + j] =
                alpha * (S0[(size_t)i * V + j] - beta * kn[i] * x[j]) + beta * kn[i] * vr[j];
    for (int j = 0; j < V; ++j) {
        double acc = 0.0;
        for (int i = 0; i < K; ++i) acc += qn[i] * S1[(size_t)i * V + j];
        o[j] = scale * acc;
    }
    /* RMSNormGated(o, z): normalise o over V, multiply by gamma, gate by SiLU(z).
     * Order and eps are this oracle's reading; the pages state neither. */
    double ms = 0.0;
    for (int j = 0; j < V; ++j) ms += o[j] * o[j];
    ms /= (double)V;
    const double rr = 1.0 / sqrt(ms + c->eps_rms);
    for (int j = 0; j < V; ++j) {
        const double silu = zr[j] * sigmoid(zr[j]);
        y[j] = o[j] * rr * c->norm_weight[j] * silu;
    }
    free(qn); free(kn); free(x); free(o);
}

/* state_out must not alias state_in: S1 is written while S0 is still being read. */
int gdn_oracle_decode_step(const double* q, const double* k, const double* v, const double* b,
                           const double* a, const double* A_log, const double* dt_bias,
                           const double* z, const double* norm_weight, const double* state_in,
                           int BH, int num_v_heads, int K, int V, double eps_l2, double eps_rms,
                           double* out, double* state_out, int nthreads) {
    if (BH < 0 || num_v_heads <= 0 || K <= 0 || V <= 0 || BH % num_v_heads != 0) return -1;
    if (state_in == state_out) return -1;
    decode_ctx c = {q, k, v, b, a, A_log, dt_bias, z, norm_weight, state_in,
                    BH, num_v_heads, K, V, eps_l2, eps_rms, out, state_out};
    for_each_unit(decode_unit, &c, (long)BH, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* gdn_oracle_conv1d_decode -- one decode token through the depthwise causal    */
/* convolution ("GDN Block TKG Kernel API Reference": gdn_conv1d_decode, conv +  */
/* silu + slide-window state; conv_weight [conv_dim, K_win], conv_state          */
/* [B, conv_dim, K_win]).                                                        */
/*                                                                              */
/* The page names the operation and the shapes only. Reading (plainest causal   */
/* depthwise convolution of width K_win over a window of the K_win latest       */
/* inputs): per batch b and channel c,                                          */
/*     window' = (state[1], ..., state[K_win-1], x)     (oldest first)          */
/*     y       = silu( sum_w weight[c][w] * window'[w] ),  silu(s) = s / (1+e^-s)*/
/*     state'  = window'                                                         */
/* No bias. Pinned by impulse responses, shift-register and pass-through cases.  */
/* ------------------------------------------------------------------------ */
int gdn_oracle_conv1d_decode(const double* x, const double* weight, const double* state_in,
                             int B, int C, int K_win, double* y, double* state_out) {
    if (B < 0 || C <= 0 || K_win <= 0) return -1;
    if (state_in == state_out) return -1;
    for (long b = 0; b < B; ++b) {
        for (long c = 0; c < C; ++c) {
            const double* s = state_in + ((size_t)b * C + c) * K_win;
            double* so = state_out + ((size_t)b * C + c) * K_win;
            for (int w = 0; w + 1 < K_win; ++w) so[w] = s[w + 1];
            so[K_win - 1] = x[(size_t)b * C + c];
            double acc = 0.0;
            for (int w = 0; w < K_win; ++w) acc += weight[(size_t)c * K_win + w] * so[w];
            y[(size_t)b * C + c] = acc / (1.0 + exp(-acc));
        }
    }
    return 0;
}
