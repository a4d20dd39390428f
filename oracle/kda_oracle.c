/*
 * Plain fp64 CPU oracle for the Kimi Delta Attention (KDA) layer core.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the reference against which the
 * CUDA library is checked.  Only the test-suite, the smoke entry point and the
 * benchmark's CPU-baseline leg may build, load or call it.  It shares no code,
 * header, table or helper with the CUDA library, and the library never calls
 * it: there is no CPU fallback.
 *
 * Every routine is the plain definition written out with sequential loops in
 * double precision.  There is no chunking, blocking, fusion or reordering.
 * The only parallelism is across independent (sequence, head) units or rows,
 * which cannot change any result.
 *
 * Sources (the web pages that define the method):
 *   [KDA-layer]   "Kimi K3 · KDA layer" (OpenModelAtlas), the KDA equation list.
 *   [SGLang]      "Kimi K3: Architecture and SGLang Day-0 Support",
 *                 section "Math details: how KDA gates and rewrites the same S".
 *   [Inside-K3]   "Inside Kimi K3: How KDA, AttnRes, and 896 Experts Work",
 *                 sections "KDA writes corrections into a recurrent matrix" and
 *                 "Short convolutions give KDA local order before recurrence".
 *   [Arch-K3]     "Kimi K3's Architecture: Kimi Delta Attention, Attention
 *                 Residuals, and 896 Experts", sections "Deriving the delta rule"
 *                 and "Channel-wise decay, and the floor K3 puts under it".
 *
 * Layouts (all row-major, C-contiguous):
 *   token tensors  [t][h][i]     t in [0, T), h in [0, H), i channel
 *   state          [n][h][j][c]  j = key channel (row), c = value channel;
 *                                Diag(alpha) scales row j [SGLang].
 *   cu_seqlens     [N+1]         sequence n owns tokens [cu[n], cu[n+1]).
 *
 * Readings of points the pages leave open are stated at each routine.
 * Return value: 0 on success, -1 on an invalid argument.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* A tiny static work splitter: unit u goes to thread u % n_threads.         */
/* ------------------------------------------------------------------------ */
typedef void (*unit_fn)(void *ctx, long unit);
typedef struct {
    unit_fn fn;
    void *ctx;
    long n_units;
    int n_threads;
    int tid;
} worker_arg;

static void *worker_main(void *p) {
    worker_arg *w = (worker_arg *)p;
    for (long u = w->tid; u < w->n_units; u += w->n_threads) w->fn(w->ctx, u);
    return NULL;
}

static void run_units(unit_fn fn, void *ctx, long n_units, int n_threads) {
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    if (n_threads == 1 || n_units <= 1) {
        for (long u = 0; u < n_units; ++u) fn(ctx, u);
        return;
    }
    pthread_t th[256];
    worker_arg args[256];
    for (int i = 0; i < n_threads; ++i) {
        args[i].fn = fn; args[i].ctx = ctx; args[i].n_units = n_units;
        args[i].n_threads = n_threads; args[i].tid = i;
        pthread_create(&th[i], NULL, worker_main, &args[i]);
    }
    for (int i = 0; i < n_threads; ++i) pthread_join(th[i], NULL);
}

/* ------------------------------------------------------------------------ */
/* One KDA token step on a d_k x d_v state, in place.                        */
/*                                                                          */
/* [KDA-layer]: S <- Diag(alpha) S;  S <- S + beta k (v - S^T k)^T;          */
/*              o~ = S^T q / sqrt(128)   (the scale is a parameter here).    */
/* [SGLang]: "gate first", then the prediction r_old is read from the        */
/* decayed state, then the delta write, then the readout of the UPDATED S.   */
/* [Inside-K3] lists the same five steps (decay, predict, error, write,      */
/* read).  alpha = exp(log_alpha); log_alpha = -inf gives alpha = 0.         */
/* ------------------------------------------------------------------------ */
static void kda_token_step(int dk, int dv, double *S, const double *q,
                           const double *k, const double *v,
                           const double *log_alpha, double beta, double scale,
                           double *o, double *r /* scratch [dv] */) {
    /* 1. decay: row j of S is multiplied by alpha_j */
    for (int j = 0; j < dk; ++j) {
        double a = exp(log_alpha[j]);
        for (int c = 0; c < dv; ++c) S[j * dv + c] *= a;
    }
    /* 2. prediction of the decayed state for key k: r = S^T k */
    for (int c = 0; c < dv; ++c) r[c] = 0.0;
    for (int j = 0; j < dk; ++j)
        for (int c = 0; c < dv; ++c) r[c] += S[j * dv + c] * k[j];
    /* 3+4. error v - r, written along k with strength beta */
    for (int j = 0; j < dk; ++j)
        for (int c = 0; c < dv; ++c) S[j * dv + c] += beta * k[j] * (v[c] - r[c]);
    /* 5. readout of the updated state with q */
    for (int c = 0; c < dv; ++c) {
        double acc = 0.0;
        for (int j = 0; j < dk; ++j) acc += S[j * dv + c] * q[j];
        o[c] = scale * acc;
    }
}

/* ------------------------------------------------------------------------ */
/* Prefill: the token-by-token recurrence over packed variable-length        */
/* sequences.  Each sequence n starts from S0[n] (zeros if S0 is NULL) and   */
/* its state after its last token is written to S_final[n] (if non-NULL).    */
/* A zero-length sequence writes no output and S_final[n] = S0[n].           */
/* ------------------------------------------------------------------------ */
typedef struct {
    int n_seqs, n_heads, dk, dv;
    const int32_t *cu;
    const double *q, *k, *v, *la, *beta, *S0;
    double scale;
    double *o, *S_final;
} prefill_ctx;

static void prefill_unit(void *p, long unit) {
    prefill_ctx *c = (prefill_ctx *)p;
    const int H = c->n_heads, dk = c->dk, dv = c->dv;
    const long n = unit / H, h = unit % H;
    double *S = (double *)malloc(sizeof(double) * (size_t)dk * dv);
    double *r = (double *)malloc(sizeof(double) * (size_t)dv);
    const size_t sdim = (size_t)dk * dv;
    if (c->S0) memcpy(S, c->S0 + ((size_t)n * H + h) * sdim, sizeof(double) * sdim);
    else memset(S, 0, sizeof(double) * sdim);
    for (long t = c->cu[n]; t < c->cu[n + 1]; ++t) {
        const size_t tk = ((size_t)t * H + h) * dk, tv = ((size_t)t * H + h) * dv;
        kda_token_step(dk, dv, S, c->q + tk, c->k + tk, c->v + tv, c->la + tk,
                       c->beta[(size_t)t * H + h], c->scale, c->o + tv, r);
    }
    if (c->S_final) memcpy(c->S_final + ((size_t)n * H + h) * sdim, S, sizeof(double) * sdim);
    free(S);
    free(r);
}

int oracle_kda_prefill(int n_seqs, int n_heads, int dk, int dv, const int32_t *cu_seqlens,
                       const double *q, const double *k, const double *v,
                       const double *log_alpha, const double *beta, const double *S0,
                       double scale, double *o, double *S_final, int n_threads) {
    if (n_seqs < 0 || n_heads <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens) return -1;
    if (cu_seqlens[0] != 0) return -1;
    for (int n = 0; n < n_seqs; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
    prefill_ctx c = {n_seqs, n_heads, dk, dv, cu_seqlens, q, k, v, log_alpha, beta, S0,
                     scale, o, S_final};
    run_units(prefill_unit, &c, (long)n_seqs * n_heads, n_threads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Decode: one token per request, state updated in place.                    */
/* It is exactly one step of the recurrence above [SGLang]: "each step reads */
/* and writes only S".                                                       */
/* ------------------------------------------------------------------------ */
typedef struct {
    int n_heads, dk, dv;
    const double *q, *k, *v, *la, *beta;
    double *S;
    double scale;
    double *o;
} decode_ctx;

static void decode_unit(void *p, long unit) {
    decode_ctx *c = (decode_ctx *)p;
    const int dk = c->dk, dv = c->dv;
    double *r = (double *)malloc(sizeof(double) * (size_t)dv);
    kda_token_step(dk, dv, c->S + (size_t)unit * dk * dv, c->q + (size_t)unit * dk,
                   c->k + (size_t)unit * dk, c->v + (size_t)unit * dv,
                   c->la + (size_t)unit * dk, c->beta[unit], c->scale,
                   c->o + (size_t)unit * dv, r);
    free(r);
}

int oracle_kda_decode_step(int batch, int n_heads, int dk, int dv, const double *q,
                           const double *k, const double *v, const double *log_alpha,
                           const double *beta, double *S_inout, double scale, double *o,
                           int n_threads) {
    if (batch < 0 || n_heads <= 0 || dk <= 0 || dv <= 0) return -1;
    decode_ctx c = {n_heads, dk, dv, q, k, v, log_alpha, beta, S_inout, scale, o};
    run_units(decode_unit, &c, (long)batch * n_heads, n_threads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Front end [KDA-layer], [Inside-K3] "Short convolutions ...":              */
/*   x^c_t = SiLU( sum_{j=0..3} w_j (.) x^p_{t-j} )   for x in {q, k, v}     */
/*   q^ = q^c / ||q^c||_2,  k^ = k^c / ||k^c||_2  (per head, 128 channels)   */
/*   log alpha = -5 sigma( e^{A_h} (z + b_alpha) )    [KDA-layer], [Arch-K3] */
/*   beta = sigma(w)                                                          */
/* Readings:                                                                  */
/*   - the conv is depthwise (the (.) product), tap j = 0 multiplies the      */
/*     current token, there is no bias, and tokens before the start of the    */
/*     token's own sequence count as zero;                                    */
/*   - conv_w is [3][H*d][4]: stream s (0 = q, 1 = k, 2 = v), channel         */
/*     h*d + i, tap j;                                                        */
/*   - the L2 norm is x * (sum x^2 + l2_eps)^(-1/2) (l2_eps = 1e-6 by         */
/*     default; the pages print no epsilon);                                  */
/*   - A is one scalar per head, b_alpha is [H][d].                           */
/* ------------------------------------------------------------------------ */
static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }
static double silu(double x) { return x * sigmoid(x); }

typedef struct {
    int n_seqs, n_heads, d;
    const int32_t *cu;
    const double *xp[3];
    const double *conv_w, *z, *A, *b, *beta_logit;
    double l2_eps;
    double *xout[3];
    double *log_alpha, *beta;
    const int32_t *seq_of_token;
} frontend_ctx;

static void frontend_token(void *p, long t) {
    frontend_ctx *c = (frontend_ctx *)p;
    const int H = c->n_heads, d = c->d;
    const long start = c->cu[c->seq_of_token[t]];
    for (int h = 0; h < H; ++h) {
        for (int s = 0; s < 3; ++s) {
            double *out = c->xout[s] + ((size_t)t * H + h) * d;
            for (int i = 0; i < d; ++i) {
                const long ch = (long)h * d + i;
                const double *w = c->conv_w + ((size_t)s * H * d + ch) * 4;
                double acc = 0.0;
                for (int j = 0; j < 4; ++j) {
                    long tj = t - j;
                    if (tj < start) break; /* zero history before the sequence */
                    acc += w[j] * c->xp[s][((size_t)tj * H + h) * d + i];
                }
                out[i] = silu(acc);
            }
            if (s < 2) { /* q and k are L2-normalised per head; v is not */
                double ss = 0.0;
                for (int i = 0; i < d; ++i) ss += out[i] * out[i];
                double inv = 1.0 / sqrt(ss + c->l2_eps);
                for (int i = 0; i < d; ++i) out[i] *= inv;
            }
        }
        const double eA = exp(c->A[h]);
        for (int i = 0; i < d; ++i) {
            const size_t idx = ((size_t)t * H + h) * d + i;
            c->log_alpha[idx] = -5.0 * sigmoid(eA * (c->z[idx] + c->b[(size_t)h * d + i]));
        }
        c->beta[(size_t)t * H + h] = sigmoid(c->beta_logit[(size_t)t * H + h]);
    }
}

int oracle_kda_frontend(int n_seqs, int n_heads, int d, const int32_t *cu_seqlens,
                        const double *qp, const double *kp, const double *vp,
                        const double *conv_w, const double *z, const double *A,
                        const double *b, const double *beta_logit, double l2_eps,
                        double *q_hat, double *k_hat, double *v_out, double *log_alpha,
                        double *beta, int n_threads) {
    if (n_seqs < 0 || n_heads <= 0 || d <= 0 || !cu_seqlens || cu_seqlens[0] != 0) return -1;
    for (int n = 0; n < n_seqs; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
    const long T = cu_seqlens[n_seqs];
    int32_t *seq_of = (int32_t *)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
    for (int n = 0; n < n_seqs; ++n)
        for (long t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) seq_of[t] = n;
    frontend_ctx c;
    c.n_seqs = n_seqs; c.n_heads = n_heads; c.d = d; c.cu = cu_seqlens;
    c.xp[0] = qp; c.xp[1] = kp; c.xp[2] = vp;
    c.conv_w = conv_w; c.z = z; c.A = A; c.b = b; c.beta_logit = beta_logit;
    c.l2_eps = l2_eps;
    c.xout[0] = q_hat; c.xout[1] = k_hat; c.xout[2] = v_out;
    c.log_alpha = log_alpha; c.beta = beta; c.seq_of_token = seq_of;
    run_units(frontend_token, &c, T, n_threads);
    free(seq_of);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Output gate [KDA-layer]: o^g = sigma(g) (.) RMSNorm(o~).                  */
/* Readings: RMSNorm is taken per head over its d channels,                  */
/*   RMSNorm(x) = x / sqrt(mean(x^2) + eps), with unit weight (no trained    */
/*   weights exist here) and eps = 1e-6 by default.                          */
/* ------------------------------------------------------------------------ */
typedef struct {
    int d;
    const double *ot, *g;
    double eps;
    double *out;
} gate_ctx;

static void gate_row(void *p, long row) {
    gate_ctx *c = (gate_ctx *)p;
    const int d = c->d;
    const double *x = c->ot + (size_t)row * d;
    const double *g = c->g + (size_t)row * d;
    double ms = 0.0;
    for (int i = 0; i < d; ++i) ms += x[i] * x[i];
    ms /= d;
    const double inv = 1.0 / sqrt(ms + c->eps);
    for (int i = 0; i < d; ++i) c->out[(size_t)row * d + i] = sigmoid(g[i]) * x[i] * inv;
}

int oracle_kda_output_gate(long n_rows, int d, const double *o_tilde, const double *g,
                           double eps, double *out, int n_threads) {
    if (n_rows < 0 || d <= 0) return -1;
    gate_ctx c = {d, o_tilde, g, eps, out};
    run_units(gate_row, &c, n_rows, n_threads);
    return 0;
}
