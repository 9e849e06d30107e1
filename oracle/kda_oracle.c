/*
 * KDA oracle: a plain, sequential, double-precision CPU statement of the
 * Kimi Delta Attention forward and of its input prologue.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA path and must never be used as a
 * fallback for it.
 *
 * What is computed (per sequence n and head h, tokens t in order):
 *
 *     S <- Diag(exp(g_t)) S                      channel-wise decay: row c of S
 *                                                 (key channel c) is scaled by
 *                                                 exp(g_t[c])
 *     S <- S - beta_t k_t (k_t^T S) + beta_t k_t v_t^T      delta-rule update
 *     o_t = scale * S^T q_t                      read-out from the updated state
 *
 * with S a K x V matrix, S_0 the caller's initial state (or zero) and the final
 * S returned as the final state.  Sources:
 *   - "ISEEKYAN/k3" README (page 1): KDA is a recurrence computed by the K3
 *     primitive, with a bounded CPU recurrence as the correctness path.
 *   - "NeMo AutoModel draft_kimi_k3" (page 2), module description: positional
 *     information reaches attention through the interleaved KDA recurrence.
 *   - "kimi-k3-mlx" review (page 3), section "The A_log shape mismatch ...":
 *     the gate g has shape (B,T,96,128) and A_log has 128 entries broadcast on
 *     the trailing head_dim axis, so the decay is per channel and shared by all
 *     heads; dt_bias has 96*128 entries.
 *   - "kimi-k3-mlx" review, section "Attention is 93 layers ...": short
 *     convolution with kernel size 4 on q, k and v, low-rank forget gate,
 *     gate_lower_bound = -5.0, 96 heads of head_dim 128.
 * The update order (decay, then delta rule, then read-out) and the recurrence
 * itself are the project's statement of the method; the pages name KDA but do
 * not print its equations.
 *
 * Layouts (all row-major, element counts not bytes):
 *   q, k, g   [Ttot, H, K]      v, o  [Ttot, H, V]      beta [Ttot, H]
 *   states    [N, H, K, V]      cu_seqlens [N + 1], cu_seqlens[0] = 0,
 *                               cu_seqlens[N] = Ttot, non-decreasing.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Recurrence                                                                 */
/* ------------------------------------------------------------------------- */

typedef struct {
    const double *q, *k, *v, *g, *beta, *s0;
    const int64_t *cu;
    int64_t N, H, K, V;
    double scale;
    double *o, *sT;
    int tid, nthreads;
    int status;
} rec_job;

/* One (sequence, head) chain, token by token. */
static void run_chain(const rec_job *j, int64_t n, int64_t h, double *S, double *kS)
{
    const int64_t H = j->H, K = j->K, V = j->V;
    if (j->s0)
        memcpy(S, j->s0 + ((n * H + h) * K) * V, sizeof(double) * K * V);
    else
        memset(S, 0, sizeof(double) * K * V);

    for (int64_t t = j->cu[n]; t < j->cu[n + 1]; ++t) {
        const double *qt = j->q + (t * H + h) * K;
        const double *kt = j->k + (t * H + h) * K;
        const double *gt = j->g + (t * H + h) * K;
        const double *vt = j->v + (t * H + h) * V;
        const double bt = j->beta[t * H + h];

        /* S <- Diag(exp(g_t)) S : key channel c scales row c. */
        for (int64_t c = 0; c < K; ++c) {
            const double a = exp(gt[c]);
            for (int64_t x = 0; x < V; ++x) S[c * V + x] *= a;
        }
        /* kS = k_t^T S  (a row vector of length V). */
        for (int64_t x = 0; x < V; ++x) kS[x] = 0.0;
        for (int64_t c = 0; c < K; ++c)
            for (int64_t x = 0; x < V; ++x) kS[x] += kt[c] * S[c * V + x];
        /* S <- S - beta k (k^T S) + beta k v^T. */
        for (int64_t c = 0; c < K; ++c)
            for (int64_t x = 0; x < V; ++x)
                S[c * V + x] = S[c * V + x] - bt * kt[c] * kS[x] + bt * kt[c] * vt[x];
        /* o_t = scale * S^T q_t. */
        double *ot = j->o + (t * H + h) * V;
        for (int64_t x = 0; x < V; ++x) {
            double acc = 0.0;
            for (int64_t c = 0; c < K; ++c) acc += S[c * V + x] * qt[c];
            ot[x] = j->scale * acc;
        }
    }
    if (j->sT) memcpy(j->sT + ((n * H + h) * K) * V, S, sizeof(double) * K * V);
}

static void *rec_worker(void *arg)
{
    rec_job *j = (rec_job *)arg;
    double *S = (double *)malloc(sizeof(double) * j->K * j->V);
    double *kS = (double *)malloc(sizeof(double) * j->V);
    if (!S || !kS) {
        j->status = -2;
        free(S);
        free(kS);
        return NULL;
    }
    const int64_t items = j->N * j->H;
    for (int64_t it = j->tid; it < items; it += j->nthreads) run_chain(j, it / j->H, it % j->H, S, kS);
    free(S);
    free(kS);
    return NULL;
}

static int spawn(void *(*fn)(void *), void *jobs, size_t job_size, int nthreads)
{
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th) return -2;
    int started = 0, rc = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, fn, (char *)jobs + job_size * (size_t)i) != 0) {
            rc = -3;
            break;
        }
        ++started;
    }
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    return rc;
}

/*
 * Returns 0 on success, -1 on invalid arguments, -2 on allocation failure,
 * -3 if a thread could not be started.
 */
int kda_oracle_forward(const double *q, const double *k, const double *v, const double *g,
                       const double *beta, const double *initial_state, const int64_t *cu_seqlens,
                       int64_t N, int64_t H, int64_t K, int64_t V, double scale, double *o,
                       double *final_state, int nthreads)
{
    if (!q || !k || !v || !g || !beta || !cu_seqlens || !o || N < 0 || H <= 0 || K <= 0 || V <= 0)
        return -1;
    if (cu_seqlens[0] != 0) return -1;
    for (int64_t n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
    if (nthreads < 1) nthreads = 1;
    if ((int64_t)nthreads > N * H && N * H > 0) nthreads = (int)(N * H);

    rec_job *jobs = (rec_job *)calloc((size_t)nthreads, sizeof(rec_job));
    if (!jobs) return -2;
    for (int i = 0; i < nthreads; ++i) {
        rec_job j = {q, k, v, g, beta, initial_state, cu_seqlens, N, H, K, V,
                     scale, o, final_state, i, nthreads, 0};
        jobs[i] = j;
    }
    int rc = spawn(rec_worker, jobs, sizeof(rec_job), nthreads);
    for (int i = 0; i < nthreads && rc == 0; ++i)
        if (jobs[i].status) rc = jobs[i].status;
    free(jobs);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* Prologue: short convolution, L2 normalisation, forget gate                 */
/* ------------------------------------------------------------------------- */

/*
 * Causal depthwise convolution of width W over the token axis, restarted at
 * every sequence boundary ("kimi-k3-mlx" review, section "Attention is 93
 * layers ...": a short convolution with kernel size 4 on q, k and v).
 *
 *     y[t, c] = sum_{j=0}^{W-1} w[c, j] * x[t - (W-1) + j, c]
 *
 * where x[s, c] = 0 for s before the start of t's sequence, so tap w[c, W-1]
 * multiplies the current token.  act = 0: no activation; act = 1: y*sigmoid(y).
 * x, y: [Ttot, C]; w: [C, W].
 */
int kda_oracle_short_conv(const double *x, const double *w, const int64_t *cu_seqlens, int64_t N,
                          int64_t C, int64_t W, int act, double *y)
{
    if (!x || !w || !cu_seqlens || !y || C <= 0 || W <= 0 || (act != 0 && act != 1)) return -1;
    for (int64_t n = 0; n < N; ++n) {
        const int64_t b = cu_seqlens[n], e = cu_seqlens[n + 1];
        for (int64_t t = b; t < e; ++t) {
            for (int64_t c = 0; c < C; ++c) {
                double acc = 0.0;
                for (int64_t j = 0; j < W; ++j) {
                    const int64_t s = t - (W - 1) + j;
                    if (s >= b) acc += w[c * W + j] * x[s * C + c];
                }
                if (act == 1) acc = acc / (1.0 + exp(-acc));
                y[t * C + c] = acc;
            }
        }
    }
    return 0;
}

/*
 * Per-row L2 normalisation: x <- x / sqrt(sum_c x_c^2 + eps), rows of length D.
 */
int kda_oracle_l2norm(double *x, int64_t rows, int64_t D, double eps)
{
    if (!x || rows < 0 || D <= 0) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        double ss = 0.0;
        for (int64_t c = 0; c < D; ++c) ss += x[r * D + c] * x[r * D + c];
        const double inv = 1.0 / sqrt(ss + eps);
        for (int64_t c = 0; c < D; ++c) x[r * D + c] *= inv;
    }
    return 0;
}

static double softplus(double z)
{
    /* log(1 + e^z) without overflow. */
    if (z > 0.0) return z + log1p(exp(-z));
    return log1p(exp(z));
}

/*
 * Per-channel forget gate ("kimi-k3-mlx" review, sections "The A_log shape
 * mismatch ..." and "Attention is 93 layers ..."):
 *
 *     g[t, h, c] = max(lower_bound, -exp(A_log[c]) * softplus(x[t, h, c] + dt_bias[h*K + c]))
 *
 * A_log has K entries broadcast on the channel axis and shared by all heads;
 * dt_bias has H*K entries.  x, g: [Ttot, H, K].
 */
int kda_oracle_gate(const double *x, const double *A_log, const double *dt_bias, int64_t Ttot,
                    int64_t H, int64_t K, double lower_bound, double *g)
{
    if (!x || !A_log || !dt_bias || !g || Ttot < 0 || H <= 0 || K <= 0) return -1;
    for (int64_t t = 0; t < Ttot; ++t)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t c = 0; c < K; ++c) {
                const int64_t i = (t * H + h) * K + c;
                const double val = -exp(A_log[c]) * softplus(x[i] + dt_bias[h * K + c]);
                g[i] = val > lower_bound ? val : lower_bound;
            }
    return 0;
}

/*
 * Output gate of the KDA layer ("kimi-k3-mlx" review, section "Attention is 93
 * layers ...": KDA has a full-rank output gate; "NeMo AutoModel draft_kimi_k3",
 * module description: K3's norms are RMS norms with the variance in fp32 and its
 * output gates are sigmoid gates).  Per row (token, head) of length V:
 *
 *     out[v] = o[v] / sqrt(mean_v(o^2) + eps) * w[v] * sigmoid(gate[v])
 *
 * w has V entries shared by all heads (NULL: all ones).  o, gate, out: [rows, V].
 */
int kda_oracle_output_gate(const double *o, const double *gate, const double *w, int64_t rows,
                           int64_t V, double eps, double *out)
{
    if (!o || !gate || !out || rows < 0 || V <= 0 || !(eps >= 0.0)) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        double ss = 0.0;
        for (int64_t c = 0; c < V; ++c) ss += o[r * V + c] * o[r * V + c];
        const double inv = 1.0 / sqrt(ss / (double)V + eps);
        for (int64_t c = 0; c < V; ++c) {
            const double sig = 1.0 / (1.0 + exp(-gate[r * V + c]));
            out[r * V + c] = o[r * V + c] * inv * (w ? w[c] : 1.0) * sig;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Projections ahead of the gate                                              */
/* ------------------------------------------------------------------------- */

/*
 * The forget gate's input and beta from the layer input x ("kimi-k3-mlx"
 * review, "Attention is 93 layers ...": a low-rank forget gate through f_a and
 * f_b; "The A_log shape mismatch ...": b_proj is [96, H], H = 7168).  Per row
 * (token) of x [rows, D]:
 *
 *     y       = f_a x                      f_a [R, D]   (the low-rank activation, kept in fp64)
 *     gate_x  = f_b y                      f_b [HK, R]  (the input of the gate)
 *     beta    = 1 / (1 + exp(-(b_proj x))) b_proj [NH, D]
 *
 * gate_x: [rows, HK], beta: [rows, NH].  Plain loops, one row at a time.
 */
int kda_oracle_gate_proj(const double *x, const double *f_a, const double *f_b, const double *b_proj,
                         int64_t rows, int64_t D, int64_t R, int64_t HK, int64_t NH, double *gate_x,
                         double *beta)
{
    if (!x || !f_a || !f_b || !b_proj || !gate_x || !beta || rows < 0 || D <= 0 || R <= 0 || HK <= 0 ||
        NH <= 0)
        return -1;
    double *y = (double *)malloc((size_t)R * sizeof(double));
    if (!y) return -2;
    for (int64_t t = 0; t < rows; ++t) {
        const double *xt = x + t * D;
        for (int64_t i = 0; i < R; ++i) {
            double acc = 0.0;
            for (int64_t d = 0; d < D; ++d) acc += f_a[i * D + d] * xt[d];
            y[i] = acc;
        }
        for (int64_t j = 0; j < HK; ++j) {
            double acc = 0.0;
            for (int64_t i = 0; i < R; ++i) acc += f_b[j * R + i] * y[i];
            gate_x[t * HK + j] = acc;
        }
        for (int64_t h = 0; h < NH; ++h) {
            double z = 0.0;
            for (int64_t d = 0; d < D; ++d) z += b_proj[h * D + d] * xt[d];
            beta[t * NH + h] = 1.0 / (1.0 + exp(-z));
        }
    }
    free(y);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Backward of the recurrence (reverse mode, token by token)                  */
/* ------------------------------------------------------------------------- */

/*
 * Gradients of  L = <dO, o> + <dS_T, S_T>  with respect to q, k, v, g, beta and
 * the initial state, through the recurrence above (same layouts; dO [Ttot, H,
 * V], dS_T and dS_0 [N, H, K, V]).  Per token, with S' = Diag(e^{g_t}) S_{t-1},
 * a = S'^T k_t, delta = beta_t (v_t - a) and S_t = S' + k_t delta^T, the
 * reverse step from the state gradient dS (of S_t) is
 *
 *     dq_t   = scale S_t dO_t              dS    += scale q_t dO_t^T
 *     ddelta = dS^T k_t                    dk_t   = dS delta
 *     dbeta_t = ddelta . (v_t - a)         dv_t   = beta_t ddelta
 *     da     = -beta_t ddelta              dS'    = dS + k_t da^T
 *     dk_t  += S' da                       dg_t[c] = sum_x dS'[c, x] S'[c, x]
 *     dS_{t-1} = Diag(e^{g_t}) dS'
 *
 * States are recomputed forward from checkpoints every 64 tokens.
 */
typedef struct {
    const double *q, *k, *v, *g, *beta, *s0, *dO, *dST;
    const int64_t *cu;
    int64_t N, H, K, V;
    double scale;
    double *dq, *dk, *dv, *dg, *dbeta, *ds0;
    int tid, nthreads;
    int status;
} bwd_job;

enum { BWD_BLOCK = 64 };

/* One forward token: S <- Diag(e^g) S, then the delta update (kS scratch [V]). */
static void fwd_token(const double *kt, const double *gt, const double *vt, double bt, int64_t K, int64_t V,
                      double *S, double *kS)
{
    for (int64_t c = 0; c < K; ++c) {
        const double ea = exp(gt[c]);
        for (int64_t x = 0; x < V; ++x) S[c * V + x] *= ea;
    }
    for (int64_t x = 0; x < V; ++x) kS[x] = 0.0;
    for (int64_t c = 0; c < K; ++c)
        for (int64_t x = 0; x < V; ++x) kS[x] += S[c * V + x] * kt[c];
    for (int64_t c = 0; c < K; ++c)
        for (int64_t x = 0; x < V; ++x) S[c * V + x] += bt * kt[c] * (vt[x] - kS[x]);
}

static int bwd_chain(const bwd_job *j, int64_t n, int64_t h)
{
    const int64_t H = j->H, K = j->K, V = j->V, KV = K * V;
    const int64_t t0 = j->cu[n], t1 = j->cu[n + 1], T = t1 - t0;
    const int64_t nblk = (T + BWD_BLOCK - 1) / BWD_BLOCK;
    double *ckpt = (double *)malloc(sizeof(double) * KV * (size_t)(nblk > 0 ? nblk : 1));
    double *prev = (double *)malloc(sizeof(double) * KV * BWD_BLOCK);  /* S_{t-1} inside a block */
    double *S = (double *)malloc(sizeof(double) * KV);
    double *Sp = (double *)malloc(sizeof(double) * KV);
    double *dS = (double *)malloc(sizeof(double) * KV);
    double *vec = (double *)malloc(sizeof(double) * (size_t)(4 * V + K));
    if (!ckpt || !prev || !S || !Sp || !dS || !vec) {
        free(ckpt); free(prev); free(S); free(Sp); free(dS); free(vec);
        return -2;
    }
    double *kS = vec, *delta = vec + V, *ddelta = vec + 2 * V, *da = vec + 3 * V;
    (void)da;

    /* forward: the state before each block */
    if (j->s0) memcpy(S, j->s0 + (n * H + h) * KV, sizeof(double) * KV);
    else memset(S, 0, sizeof(double) * KV);
    for (int64_t b = 0; b < nblk; ++b) {
        memcpy(ckpt + b * KV, S, sizeof(double) * KV);
        const int64_t e = (b + 1) * BWD_BLOCK < T ? (b + 1) * BWD_BLOCK : T;
        for (int64_t t = t0 + b * BWD_BLOCK; t < t0 + e; ++t)
            fwd_token(j->k + (t * H + h) * K, j->g + (t * H + h) * K, j->v + (t * H + h) * V,
                      j->beta[t * H + h], K, V, S, kS);
    }

    /* backward */
    if (j->dST) memcpy(dS, j->dST + (n * H + h) * KV, sizeof(double) * KV);
    else memset(dS, 0, sizeof(double) * KV);
    for (int64_t b = nblk - 1; b >= 0; --b) {
        const int64_t s = t0 + b * BWD_BLOCK;
        const int64_t e = t0 + ((b + 1) * BWD_BLOCK < T ? (b + 1) * BWD_BLOCK : T);
        memcpy(S, ckpt + b * KV, sizeof(double) * KV);
        for (int64_t t = s; t < e; ++t) {
            memcpy(prev + (t - s) * KV, S, sizeof(double) * KV);
            fwd_token(j->k + (t * H + h) * K, j->g + (t * H + h) * K, j->v + (t * H + h) * V,
                      j->beta[t * H + h], K, V, S, kS);
        }
        for (int64_t t = e - 1; t >= s; --t) {
            const double *qt = j->q + (t * H + h) * K, *kt = j->k + (t * H + h) * K;
            const double *gt = j->g + (t * H + h) * K, *vt = j->v + (t * H + h) * V;
            const double *dot = j->dO + (t * H + h) * V;
            const double bt = j->beta[t * H + h];
            double *dqt = j->dq + (t * H + h) * K, *dkt = j->dk + (t * H + h) * K;
            double *dvt = j->dv + (t * H + h) * V, *dgt = j->dg + (t * H + h) * K;
            /* S' = Diag(e^g) S_{t-1}; a = S'^T k; delta = beta (v - a); S_t = S' + k delta^T */
            const double *Sprev = prev + (t - s) * KV;
            for (int64_t c = 0; c < K; ++c) {
                const double ea = exp(gt[c]);
                for (int64_t x = 0; x < V; ++x) Sp[c * V + x] = ea * Sprev[c * V + x];
            }
            for (int64_t x = 0; x < V; ++x) {
                double acc = 0.0;
                for (int64_t c = 0; c < K; ++c) acc += kt[c] * Sp[c * V + x];
                kS[x] = acc;
                delta[x] = bt * (vt[x] - acc);
            }
            /* dq = scale S_t dO  (S_t = S' + k delta^T) */
            for (int64_t c = 0; c < K; ++c) {
                double acc = 0.0;
                for (int64_t x = 0; x < V; ++x) acc += (Sp[c * V + x] + kt[c] * delta[x]) * dot[x];
                dqt[c] = j->scale * acc;
            }
            /* dS += scale q dO^T */
            for (int64_t c = 0; c < K; ++c)
                for (int64_t x = 0; x < V; ++x) dS[c * V + x] += j->scale * qt[c] * dot[x];
            /* ddelta = dS^T k;  dk = dS delta */
            for (int64_t x = 0; x < V; ++x) {
                double acc = 0.0;
                for (int64_t c = 0; c < K; ++c) acc += dS[c * V + x] * kt[c];
                ddelta[x] = acc;
            }
            for (int64_t c = 0; c < K; ++c) {
                double acc = 0.0;
                for (int64_t x = 0; x < V; ++x) acc += dS[c * V + x] * delta[x];
                dkt[c] = acc;
            }
            /* dbeta = ddelta . (v - a); dv = beta ddelta; da = -beta ddelta */
            double db = 0.0;
            for (int64_t x = 0; x < V; ++x) {
                db += ddelta[x] * (vt[x] - kS[x]);
                dvt[x] = bt * ddelta[x];
            }
            j->dbeta[t * H + h] = db;
            /* dS' = dS + k da^T (in place); dk += S' da; dg = rowsum(dS' * S') */
            for (int64_t c = 0; c < K; ++c) {
                double acc = 0.0;
                for (int64_t x = 0; x < V; ++x) acc += Sp[c * V + x] * (-bt * ddelta[x]);
                dkt[c] += acc;
            }
            for (int64_t c = 0; c < K; ++c) {
                double acc = 0.0;
                const double ea = exp(gt[c]);
                for (int64_t x = 0; x < V; ++x) {
                    const double d = dS[c * V + x] + kt[c] * (-bt * ddelta[x]);
                    acc += d * Sp[c * V + x];
                    dS[c * V + x] = ea * d; /* dS_{t-1} = Diag(e^g) dS' */
                }
                dgt[c] = acc;
            }
        }
    }
    if (j->ds0) memcpy(j->ds0 + (n * H + h) * KV, dS, sizeof(double) * KV);
    free(ckpt); free(prev); free(S); free(Sp); free(dS); free(vec);
    return 0;
}

static void *bwd_worker(void *arg)
{
    bwd_job *j = (bwd_job *)arg;
    const int64_t items = j->N * j->H;
    for (int64_t it = j->tid; it < items; it += j->nthreads) {
        const int rc = bwd_chain(j, it / j->H, it % j->H);
        if (rc) { j->status = rc; break; }
    }
    return NULL;
}

/* Returns 0, -1 (invalid arguments), -2 (allocation) or -3 (threads). */
int kda_oracle_backward(const double *q, const double *k, const double *v, const double *g,
                        const double *beta, const double *initial_state, const int64_t *cu_seqlens,
                        int64_t N, int64_t H, int64_t K, int64_t V, double scale, const double *dO,
                        const double *dST, double *dq, double *dk, double *dv, double *dg, double *dbeta,
                        double *ds0, int nthreads)
{
    if (!q || !k || !v || !g || !beta || !cu_seqlens || !dO || !dq || !dk || !dv || !dg || !dbeta ||
        N < 0 || H <= 0 || K <= 0 || V <= 0)
        return -1;
    if (cu_seqlens[0] != 0) return -1;
    for (int64_t n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
    if (nthreads < 1) nthreads = 1;
    if ((int64_t)nthreads > N * H && N * H > 0) nthreads = (int)(N * H);
    bwd_job *jobs = (bwd_job *)calloc((size_t)nthreads, sizeof(bwd_job));
    if (!jobs) return -2;
    for (int i = 0; i < nthreads; ++i) {
        bwd_job jb = {q, k, v, g, beta, initial_state, dO, dST, cu_seqlens, N, H, K, V, scale,
                      dq, dk, dv, dg, dbeta, ds0, i, nthreads, 0};
        jobs[i] = jb;
    }
    int rc = spawn(bwd_worker, jobs, sizeof(bwd_job), nthreads);
    for (int i = 0; i < nthreads && rc == 0; ++i)
        if (jobs[i].status) rc = jobs[i].status;
    free(jobs);
    return rc;
}
