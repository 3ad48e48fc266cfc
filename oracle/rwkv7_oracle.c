/*
 * rwkv7_oracle.c -- plain, slow CPU oracle of the RWKV-7 batched decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  It shares no code, header or table
 * with the CUDA path.
 *
 * What it computes (sources):
 *  - The decode step of an RWKV-7 ("x070") model for one token of one sequence:
 *    the path the RWKV-Server article ("RWKV 批量推理中 Prefill 的正确打开方式",
 *    §三, B>1/T=1 decode path) and the RWKV-Runner Albatross article
 *    ("连续批处理Worker 主循环": forward_seq_batch, sample_next_tokens_batch) run
 *    per slot.  The pages print no equations; the public RWKV-7 definition is
 *    taken as the plain reading: LayerNorm + token-shift mixes, r/k/v
 *    projections, LoRA gates, the 64x64 per-head state update, GroupNorm, bonus
 *    term, output gate, then the ReLU^2 channel mix.
 *  - A chunked prefill (layer-major over a block of tokens, with the state
 *    transition written as explicit dense 64x64 matrices and chained products).
 *    It is a second formulation of the same recurrence, used to check the
 *    stepwise one (the prefill/decode split of the RWKV-Server article, §五).
 *  - The sampler: presence/frequency penalty with decaying occurrence counts,
 *    top-p / top-k / temperature, one Philox4x32-10 draw (Salmon et al., SC'11,
 *    "Parallel Random Numbers: As Easy as 1, 2, 3").  Defaults and the penalty
 *    come from the Albatross adapter and worker loop sections.
 *
 * Precision: every model quantity is fp64, except that the values the method
 * feeds to its fp16 matrix products (the six token-shift mixes, the channel-mix
 * input, the LoRA hidden vectors, the gated attention output, the ReLU^2 hidden
 * vector and the final LayerNorm output) are rounded to fp16 first, because the
 * pages' kernels run fp16 weights ("CUDA fp16" model; *_f16 kernels).  The
 * sampler works in fp32 and integers: its float steps decide integers, and both
 * sides take those decisions in fp32 with the same operations.
 *
 * Build: gcc -O2 -fPIC -shared -fopenmp -ffp-contract=off (no fast-math).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_N 64 /* head size */

/* ------------------------------------------------------------------------- */
/* IEEE binary16 <-> binary64.                                                */
/* ------------------------------------------------------------------------- */

/* Exact decode of a binary16 bit pattern. */
double orc_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24); /* zero or subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* Round a double to the nearest binary16 (ties to even). */
uint16_t orc_f64_to_f16(double x) {
    uint16_t sign = (uint16_t)(signbit(x) ? 0x8000u : 0u);
    double a = fabs(x);
    if (isnan(x)) return (uint16_t)(sign | 0x7e00u);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) -> unbiased exponent e-1 */
    int ub = e - 1;
    if (ub < -14) {
        /* subnormal range: value = q * 2^-24, q integer after rounding */
        double q = rint(ldexp(a, 24)); /* exact scaling, then RNE */
        return (uint16_t)(sign | (uint16_t)q); /* q == 1024 rolls into the smallest normal */
    }
    double q = rint(ldexp(a, 10 - ub)); /* mantissa with implicit bit, in [1024, 2048] */
    if (q >= 2048.0) {
        q = 1024.0;
        ub += 1;
    }
    if (ub > 15) return (uint16_t)(sign | 0x7c00u); /* overflow -> inf */
    return (uint16_t)(sign | (uint16_t)((ub + 15) << 10) | (uint16_t)((int)q - 1024));
}

static double f16_lut[65536];
static int f16_lut_ready = 0;

static void build_lut(void) {
    if (f16_lut_ready) return;
    for (int i = 0; i < 65536; ++i) f16_lut[i] = orc_f16_to_f64((uint16_t)i);
    f16_lut_ready = 1;
}

static inline double H(uint16_t h) { return f16_lut[h]; }
static inline double R16(double x) { return H(orc_f64_to_f16(x)); }

/* ------------------------------------------------------------------------- */
/* Primitives.                                                                */
/* ------------------------------------------------------------------------- */

static int g_threads = 1;

void orc_set_threads(int n) {
    g_threads = n < 1 ? 1 : n;
#ifdef _OPENMP
    omp_set_num_threads(g_threads);
#endif
}

int orc_get_threads(void) { return g_threads; }

/* y[o] = sum_i W[o][i] x[i]; W is fp16 [rows][cols] with a row per output. */
void orc_gemv(int rows, int cols, const uint16_t *W, const double *x, double *y) {
    build_lut();
#pragma omp parallel for schedule(static) if (rows >= 256)
    for (int o = 0; o < rows; ++o) {
        const uint16_t *w = W + (size_t)o * cols;
        double acc = 0.0;
        for (int i = 0; i < cols; ++i) acc += H(w[i]) * x[i];
        y[o] = acc;
    }
}

/* The int8 weight variant: a matrix is given as int8 values q [rows][cols] and
 * one fp16 scale per row, and stands for W[o][i] = q[o][i] * scale[o].
 * y[o] = scale[o] * sum_i q[o][i] x[i] (the scale factored out of the row sum). */
void orc_gemv_i8(int rows, int cols, const int8_t *q, const uint16_t *scale, const double *x, double *y) {
    build_lut();
#pragma omp parallel for schedule(static) if (rows >= 256)
    for (int o = 0; o < rows; ++o) {
        const int8_t *w = q + (size_t)o * cols;
        double acc = 0.0;
        for (int i = 0; i < cols; ++i) acc += (double)w[i] * x[i];
        y[o] = H(scale[o]) * acc;
    }
}

/* LayerNorm over n values: (x - mean) / sqrt(var + eps) * g + b, biased variance. */
void orc_layernorm(int n, const double *x, const double *g, const double *b, double eps,
                   double *y) {
    double mean = 0.0;
    for (int i = 0; i < n; ++i) mean += x[i];
    mean /= n;
    double var = 0.0;
    for (int i = 0; i < n; ++i) var += (x[i] - mean) * (x[i] - mean);
    var /= n;
    double rs = 1.0 / sqrt(var + eps);
    for (int i = 0; i < n; ++i) y[i] = (x[i] - mean) * rs * g[i] + b[i];
}

/* GroupNorm: LayerNorm of each consecutive group of `gsize` values, with the
 * affine parameters indexed over the whole vector. */
void orc_groupnorm(int n, int gsize, const double *x, const double *g, const double *b,
                   double eps, double *y) {
    for (int s = 0; s < n; s += gsize) orc_layernorm(gsize, x + s, g + s, b + s, eps, y + s);
}

static inline double sigm(double x) { return 1.0 / (1.0 + exp(-x)); }

/*
 * One step of the per-head state update, rank-1 form.  S is N x N, row i is a
 * value index, column j a key index.
 *   sa_i     = sum_j S[i][j] kh_j
 *   S[i][j] <- S[i][j] decay_j - sa_i kh_j a_j + vp_i kp_j
 *   y_i      = sum_j S[i][j] r_j          (after the update)
 * decay and a are taken as direct inputs so that the special cases decay = 1,
 * a = 0 etc. (unreachable through the model's parametrisation) can be checked.
 */
void orc_wkv_step(int N, double *S, const double *r, const double *decay, const double *kh,
                  const double *a, const double *kp, const double *vp, double *y) {
    for (int i = 0; i < N; ++i) {
        double *Si = S + (size_t)i * N;
        double sa = 0.0;
        for (int j = 0; j < N; ++j) sa += Si[j] * kh[j];
        double yi = 0.0;
        for (int j = 0; j < N; ++j) {
            Si[j] = Si[j] * decay[j] - sa * kh[j] * a[j] + vp[i] * kp[j];
            yi += Si[j] * r[j];
        }
        y[i] = yi;
    }
}

/* Dense N x N helpers for the chunked form. */
static void mat_mul(int N, const double *A, const double *B, double *C) { /* C = A B */
    for (int i = 0; i < N; ++i)
        for (int j = 0; j < N; ++j) {
            double acc = 0.0;
            for (int m = 0; m < N; ++m) acc += A[i * N + m] * B[m * N + j];
            C[i * N + j] = acc;
        }
}

static void transition(int N, const double *decay, const double *kh, const double *a,
                       double *A) { /* A = diag(decay) - kh (a*kh)^T */
    for (int m = 0; m < N; ++m)
        for (int j = 0; j < N; ++j)
            A[m * N + j] = (m == j ? decay[j] : 0.0) - kh[m] * (a[j] * kh[j]);
}

/*
 * Chunked form over T tokens of one head.  With A_t = diag(decay_t) - kh_t (a_t*kh_t)^T
 * the recurrence is S_t = S_{t-1} A_t + vp_t kp_t^T.  Unrolled from the state S0 at
 * the start of the block:
 *   S_t = S0 P_t + sum_{s<=t} vp_s kp_s^T Q(s,t),  P_t = A_1...A_t,  Q(s,t) = A_{s+1}...A_t
 *   y_t = S_t r_t
 * Inputs are [T][N] row-major; S is updated to S_T, y is [T][N].
 */
void orc_wkv_chunk(int N, int T, double *S, const double *r, const double *decay,
                   const double *kh, const double *a, const double *kp, const double *vp,
                   double *y) {
    size_t NN = (size_t)N * N;
    double *A = malloc(sizeof(double) * NN * (size_t)T); /* all transitions */
    double *P = calloc(NN, sizeof(double));
    double *tmp = malloc(sizeof(double) * NN);
    double *g = malloc(sizeof(double) * N);
    double *g2 = malloc(sizeof(double) * N);
    double *u = malloc(sizeof(double) * N);
    for (int t = 0; t < T; ++t)
        transition(N, decay + (size_t)t * N, kh + (size_t)t * N, a + (size_t)t * N,
                   A + NN * t);
    /* outputs */
    for (size_t i = 0; i < NN; ++i) P[i] = (i % (N + 1) == 0) ? 1.0 : 0.0;
    for (int t = 0; t < T; ++t) {
        mat_mul(N, P, A + NN * t, tmp); /* P_t = P_{t-1} A_t */
        memcpy(P, tmp, sizeof(double) * NN);
        const double *rt = r + (size_t)t * N;
        /* u = P_t r_t ; y_t = S0 u */
        for (int m = 0; m < N; ++m) {
            double acc = 0.0;
            for (int j = 0; j < N; ++j) acc += P[m * N + j] * rt[j];
            u[m] = acc;
        }
        double *yt = y + (size_t)t * N;
        for (int i = 0; i < N; ++i) {
            double acc = 0.0;
            for (int m = 0; m < N; ++m) acc += S[i * N + m] * u[m];
            yt[i] = acc;
        }
        /* + sum_{s<=t} vp_s (kp_s . Q(s,t) r_t), walking s downwards with g = Q(s,t) r_t */
        memcpy(g, rt, sizeof(double) * N);
        for (int s = t; s >= 0; --s) {
            const double *kps = kp + (size_t)s * N, *vps = vp + (size_t)s * N;
            double c = 0.0;
            for (int j = 0; j < N; ++j) c += kps[j] * g[j];
            for (int i = 0; i < N; ++i) yt[i] += vps[i] * c;
            if (s > 0) { /* g <- A_s g  (Q(s-1,t) = A_s Q(s,t)) */
                const double *As = A + NN * s;
                for (int m = 0; m < N; ++m) {
                    double acc = 0.0;
                    for (int j = 0; j < N; ++j) acc += As[m * N + j] * g[j];
                    g2[m] = acc;
                }
                memcpy(g, g2, sizeof(double) * N);
            }
        }
    }
    /* final state: S_T = S0 P_T + sum_s vp_s (kp_s^T Q(s,T)); R = Q(s,T) built from the right */
    double *Snew = malloc(sizeof(double) * NN);
    double *R = malloc(sizeof(double) * NN);
    mat_mul(N, S, P, Snew);
    for (size_t i = 0; i < NN; ++i) R[i] = (i % (N + 1) == 0) ? 1.0 : 0.0;
    for (int s = T - 1; s >= 0; --s) {
        const double *kps = kp + (size_t)s * N, *vps = vp + (size_t)s * N;
        for (int j = 0; j < N; ++j) { /* row vector kp_s^T R */
            double acc = 0.0;
            for (int m = 0; m < N; ++m) acc += kps[m] * R[m * N + j];
            g[j] = acc;
        }
        for (int i = 0; i < N; ++i)
            for (int j = 0; j < N; ++j) Snew[i * N + j] += vps[i] * g[j];
        if (s > 0) { /* R <- A_s R */
            mat_mul(N, A + NN * s, R, tmp);
            memcpy(R, tmp, sizeof(double) * NN);
        }
    }
    memcpy(S, Snew, sizeof(double) * NN);
    free(A); free(P); free(tmp); free(g); free(g2); free(u); free(Snew); free(R);
}

/* ------------------------------------------------------------------------- */
/* Model.                                                                     */
/* ------------------------------------------------------------------------- */

/* Tensor order of the pointer table handed to orc_model_new. */
enum { G_EMB, G_LN0W, G_LN0B, G_LNOW, G_LNOB, G_HEAD, G_COUNT };
enum {
    T_LN1W, T_LN1B, T_LN2W, T_LN2B,
    T_XR, T_XW, T_XK, T_XV, T_XA, T_XG,
    T_W0, T_W1, T_W2, T_A0, T_A1, T_A2, T_V0, T_V1, T_V2, T_G1, T_G2,
    T_KK, T_KA, T_RK, T_WR, T_WK, T_WV, T_WO, T_LNXW, T_LNXB,
    T_FXK, T_FK, T_FV, T_COUNT
};

typedef struct {
    int L, d, N, H, F, V, rw, ra, rv, rg;
    const uint16_t *g[G_COUNT];
    const uint16_t **t; /* [L][T_COUNT] */
    const int8_t **q8;      /* [G_COUNT + L * T_COUNT]: int8 values of a matrix given in int8, else NULL */
    const uint16_t **s8;    /* its fp16 row scales */
} orc_model;

typedef struct {
    double *wkv;       /* [L][H][N][N] */
    double *shift_att; /* [L][d] */
    double *shift_ffn; /* [L][d] */
} orc_state;

int orc_tensor_count(int n_layer) { return G_COUNT + n_layer * T_COUNT; }

/* dims: L, d, head_size, F, V, rw, ra, rv, rg.  ptrs: G_COUNT globals then T_COUNT per layer. */
orc_model *orc_model_new(const int32_t *dims, const uint16_t *const *ptrs) {
    build_lut();
    if (dims[2] != ORC_N || dims[1] % ORC_N) return NULL;
    orc_model *m = calloc(1, sizeof(orc_model));
    m->L = dims[0]; m->d = dims[1]; m->N = dims[2]; m->F = dims[3]; m->V = dims[4];
    m->rw = dims[5]; m->ra = dims[6]; m->rv = dims[7]; m->rg = dims[8];
    m->H = m->d / m->N;
    for (int i = 0; i < G_COUNT; ++i) m->g[i] = ptrs[i];
    m->t = malloc(sizeof(uint16_t *) * (size_t)m->L * T_COUNT);
    for (int i = 0; i < m->L * T_COUNT; ++i) m->t[i] = ptrs[G_COUNT + i];
    m->q8 = calloc((size_t)G_COUNT + (size_t)m->L * T_COUNT, sizeof(int8_t *));
    m->s8 = calloc((size_t)G_COUNT + (size_t)m->L * T_COUNT, sizeof(uint16_t *));
    return m;
}

/* Give tensor `index` (pointer-table order) as int8 values + fp16 row scales. */
int orc_model_set_i8(orc_model *m, int index, const int8_t *q, const uint16_t *scale) {
    if (!m || index < 0 || index >= G_COUNT + m->L * T_COUNT || !q || !scale) return -1;
    m->q8[index] = q;
    m->s8[index] = scale;
    return 0;
}

void orc_model_free(orc_model *m) {
    if (!m) return;
    free(m->t);
    free(m->q8);
    free(m->s8);
    free(m);
}

static inline const uint16_t *LT(const orc_model *m, int l, int k) { return m->t[l * T_COUNT + k]; }
static inline int LI(int l, int k) { return G_COUNT + l * T_COUNT + k; }

/* y = W x for matrix tensor `index`, in whichever form it was given. */
static void mgemv(const orc_model *m, int index, int rows, int cols, const double *x, double *y) {
    if (m->q8[index])
        orc_gemv_i8(rows, cols, m->q8[index], m->s8[index], x, y);
    else
        orc_gemv(rows, cols, index < G_COUNT ? m->g[index] : m->t[index - G_COUNT], x, y);
}

static void vec16(int n, const uint16_t *p, double *out) {
    for (int i = 0; i < n; ++i) out[i] = H(p[i]);
}

size_t orc_state_doubles(const orc_model *m) {
    return (size_t)m->L * m->H * m->N * m->N + 2 * (size_t)m->L * m->d;
}

orc_state *orc_state_new(const orc_model *m) {
    orc_state *s = calloc(1, sizeof(orc_state));
    s->wkv = calloc((size_t)m->L * m->H * m->N * m->N, sizeof(double));
    s->shift_att = calloc((size_t)m->L * m->d, sizeof(double));
    s->shift_ffn = calloc((size_t)m->L * m->d, sizeof(double));
    return s;
}

void orc_state_free(orc_state *s) {
    if (!s) return;
    free(s->wkv); free(s->shift_att); free(s->shift_ffn); free(s);
}

/* Export / import: wkv [L][H][N][N], then shift_att [L][d], then shift_ffn [L][d]. */
void orc_state_get(const orc_model *m, const orc_state *s, double *out) {
    size_t nw = (size_t)m->L * m->H * m->N * m->N, ns = (size_t)m->L * m->d;
    memcpy(out, s->wkv, nw * sizeof(double));
    memcpy(out + nw, s->shift_att, ns * sizeof(double));
    memcpy(out + nw + ns, s->shift_ffn, ns * sizeof(double));
}

void orc_state_set(const orc_model *m, orc_state *s, const double *in) {
    size_t nw = (size_t)m->L * m->H * m->N * m->N, ns = (size_t)m->L * m->d;
    memcpy(s->wkv, in, nw * sizeof(double));
    memcpy(s->shift_att, in + nw, ns * sizeof(double));
    memcpy(s->shift_ffn, in + nw + ns, ns * sizeof(double));
}

/* Per-layer quantities of one token, computed from the layer input. */
typedef struct {
    double *xl, *xr, *xw, *xk, *xv, *xa, *xg;
    double *r, *k, *v, *hw, *ha, *hv, *hg, *dw, *decay, *a, *vg, *g;
    double *kh, *kp, *vp, *y, *z, *tmp;
} orc_tok;

static double *buf_take(double **pool, int n) {
    double *p = *pool;
    *pool += n;
    return p;
}

static double *tok_alloc(const orc_model *m, orc_tok *w) {
    int d = m->d, rmax = m->rw + m->ra + m->rv + m->rg;
    double *pool0 = calloc((size_t)24 * d + rmax + m->F, sizeof(double)), *p = pool0;
    w->xl = buf_take(&p, d); w->xr = buf_take(&p, d); w->xw = buf_take(&p, d);
    w->xk = buf_take(&p, d); w->xv = buf_take(&p, d); w->xa = buf_take(&p, d);
    w->xg = buf_take(&p, d); w->r = buf_take(&p, d); w->k = buf_take(&p, d);
    w->v = buf_take(&p, d); w->dw = buf_take(&p, d); w->decay = buf_take(&p, d);
    w->a = buf_take(&p, d); w->vg = buf_take(&p, d); w->g = buf_take(&p, d);
    w->kh = buf_take(&p, d); w->kp = buf_take(&p, d); w->vp = buf_take(&p, d);
    w->y = buf_take(&p, d); w->z = buf_take(&p, d);
    w->hw = buf_take(&p, m->rw); w->ha = buf_take(&p, m->ra);
    w->hv = buf_take(&p, m->rv); w->hg = buf_take(&p, m->rg);
    w->tmp = buf_take(&p, m->F > 4 * d ? m->F : 4 * d);
    return pool0;
}

/*
 * Time-mix front half for one token: LayerNorm, token shift, the six mixes,
 * projections and LoRA gates, the normalised removal key kh, the modified key
 * kp and the value vp (mixed with the layer-0 value v_first for l > 0).
 * `prev` is the previous token's LayerNorm output (the shift state).
 */
static void tmix_front(const orc_model *m, int l, const double *x, const double *prev,
                       double *v_first, orc_tok *w) {
    int d = m->d, N = m->N;
    double *gam = w->tmp, *bet = w->tmp + d, *mu = w->tmp + 2 * d;
    vec16(d, LT(m, l, T_LN1W), gam);
    vec16(d, LT(m, l, T_LN1B), bet);
    orc_layernorm(d, x, gam, bet, 1e-5, w->xl);
    const int mix_id[6] = {T_XR, T_XW, T_XK, T_XV, T_XA, T_XG};
    double *mix_out[6] = {w->xr, w->xw, w->xk, w->xv, w->xa, w->xg};
    for (int q = 0; q < 6; ++q) {
        vec16(d, LT(m, l, mix_id[q]), mu);
        for (int i = 0; i < d; ++i)
            mix_out[q][i] = R16(w->xl[i] + (prev[i] - w->xl[i]) * mu[i]);
    }
    mgemv(m, LI(l, T_WR), d, d, w->xr, w->r);
    mgemv(m, LI(l, T_WK), d, d, w->xk, w->k);
    mgemv(m, LI(l, T_WV), d, d, w->xv, w->v);
    /* LoRA down projections (fp16-rounded hidden vectors) */
    mgemv(m, LI(l, T_W1), m->rw, d, w->xw, w->hw);
    for (int j = 0; j < m->rw; ++j) w->hw[j] = R16(tanh(w->hw[j]));
    mgemv(m, LI(l, T_A1), m->ra, d, w->xa, w->ha);
    for (int j = 0; j < m->ra; ++j) w->ha[j] = R16(w->ha[j]);
    mgemv(m, LI(l, T_V1), m->rv, d, w->xv, w->hv);
    for (int j = 0; j < m->rv; ++j) w->hv[j] = R16(w->hv[j]);
    mgemv(m, LI(l, T_G1), m->rg, d, w->xg, w->hg);
    for (int j = 0; j < m->rg; ++j) w->hg[j] = R16(sigm(w->hg[j]));
    /* LoRA up projections and gates */
    double *bias = w->tmp + 3 * d;
    mgemv(m, LI(l, T_W2), d, m->rw, w->hw, w->dw);
    vec16(d, LT(m, l, T_W0), bias);
    for (int i = 0; i < d; ++i) {
        w->dw[i] += bias[i];
        /* decay = exp(-exp(-0.5) * sigmoid(w0 + LoRA_w)) in (0.545, 1) */
        w->decay[i] = exp(-exp(-0.5) * sigm(w->dw[i]));
    }
    mgemv(m, LI(l, T_A2), d, m->ra, w->ha, w->a);
    vec16(d, LT(m, l, T_A0), bias);
    for (int i = 0; i < d; ++i) w->a[i] = sigm(bias[i] + w->a[i]);
    mgemv(m, LI(l, T_V2), d, m->rv, w->hv, w->vg);
    vec16(d, LT(m, l, T_V0), bias);
    for (int i = 0; i < d; ++i) w->vg[i] = sigm(bias[i] + w->vg[i]);
    mgemv(m, LI(l, T_G2), d, m->rg, w->hg, w->g);
    /* removal key kh = normalize(k * k_k) per head; modified key kp = k * (1 + (a-1) k_a) */
    double *kk = w->tmp, *ka = w->tmp + d;
    vec16(d, LT(m, l, T_KK), kk);
    vec16(d, LT(m, l, T_KA), ka);
    for (int h = 0; h < d / N; ++h) {
        double ss = 0.0;
        for (int j = 0; j < N; ++j) {
            double t = w->k[h * N + j] * kk[h * N + j];
            ss += t * t;
        }
        double nrm = sqrt(ss);
        if (nrm < 1e-12) nrm = 1e-12;
        for (int j = 0; j < N; ++j) w->kh[h * N + j] = w->k[h * N + j] * kk[h * N + j] / nrm;
    }
    for (int i = 0; i < d; ++i) w->kp[i] = w->k[i] * (1.0 + (w->a[i] - 1.0) * ka[i]);
    if (l == 0) {
        memcpy(v_first, w->v, sizeof(double) * d);
        memcpy(w->vp, w->v, sizeof(double) * d);
    } else {
        for (int i = 0; i < d; ++i) w->vp[i] = w->v[i] + (v_first[i] - w->v[i]) * w->vg[i];
    }
}

/* Time-mix back half: GroupNorm, bonus, output gate and the output projection
 * added to the residual x. */
static void tmix_back(const orc_model *m, int l, double *x, orc_tok *w) {
    int d = m->d, N = m->N;
    double *gam = w->tmp, *bet = w->tmp + d, *rk = w->tmp + 2 * d, *o = w->tmp + 3 * d;
    vec16(d, LT(m, l, T_LNXW), gam);
    vec16(d, LT(m, l, T_LNXB), bet);
    vec16(d, LT(m, l, T_RK), rk);
    orc_groupnorm(d, N, w->y, gam, bet, 64e-5, w->z);
    for (int h = 0; h < d / N; ++h) {
        double bonus = 0.0;
        for (int j = 0; j < N; ++j) bonus += w->r[h * N + j] * w->kp[h * N + j] * rk[h * N + j];
        for (int i = 0; i < N; ++i) w->z[h * N + i] += bonus * w->vp[h * N + i];
    }
    for (int i = 0; i < d; ++i) w->z[i] = R16(w->z[i] * w->g[i]);
    mgemv(m, LI(l, T_WO), d, d, w->z, o);
    for (int i = 0; i < d; ++i) x[i] += o[i];
}

/* Channel mix: LayerNorm, token shift with one mix, ReLU^2 key, value, residual. */
static void cmix(const orc_model *m, int l, double *x, const double *prev, double *xl2_out,
                 orc_tok *w) {
    int d = m->d, F = m->F;
    double *gam = w->tmp, *bet = w->tmp + d, *mu = w->tmp + 2 * d;
    double *xk = w->xk; /* reuse */
    vec16(d, LT(m, l, T_LN2W), gam);
    vec16(d, LT(m, l, T_LN2B), bet);
    orc_layernorm(d, x, gam, bet, 1e-5, xl2_out);
    vec16(d, LT(m, l, T_FXK), mu);
    for (int i = 0; i < d; ++i) xk[i] = R16(xl2_out[i] + (prev[i] - xl2_out[i]) * mu[i]);
    double *hbuf = malloc(sizeof(double) * F), *o = malloc(sizeof(double) * d);
    mgemv(m, LI(l, T_FK), F, d, xk, hbuf);
    for (int f = 0; f < F; ++f) {
        double t = hbuf[f] > 0.0 ? hbuf[f] : 0.0;
        hbuf[f] = R16(t * t);
    }
    mgemv(m, LI(l, T_FV), d, F, hbuf, o);
    for (int i = 0; i < d; ++i) x[i] += o[i];
    free(hbuf);
    free(o);
}

static void embed(const orc_model *m, int32_t token, double *x, double *tmp) {
    int d = m->d;
    const uint16_t *e = m->g[G_EMB] + (size_t)token * d;
    double *xe = tmp, *gam = tmp + d, *bet = tmp + 2 * d;
    vec16(d, e, xe);
    vec16(d, m->g[G_LN0W], gam);
    vec16(d, m->g[G_LN0B], bet);
    orc_layernorm(d, xe, gam, bet, 1e-5, x);
}

static void head(const orc_model *m, const double *x, double *logits, double *tmp) {
    int d = m->d;
    double *gam = tmp, *bet = tmp + d, *xo = tmp + 2 * d;
    vec16(d, m->g[G_LNOW], gam);
    vec16(d, m->g[G_LNOB], bet);
    orc_layernorm(d, x, gam, bet, 1e-5, xo);
    for (int i = 0; i < d; ++i) xo[i] = R16(xo[i]);
    mgemv(m, G_HEAD, m->V, d, xo, logits);
}

/*
 * One decode step of one sequence: consume `token`, update the state, and
 * write the next-token logits (fp64, [V]) if `logits` is not NULL.
 */
int orc_step(const orc_model *m, orc_state *s, int32_t token, double *logits) {
    if (token < 0 || token >= m->V) return -1;
    int d = m->d, N = m->N, H = m->H;
    orc_tok w;
    double *pool = tok_alloc(m, &w);
    double *x = malloc(sizeof(double) * d), *v_first = malloc(sizeof(double) * d);
    double *t3 = malloc(sizeof(double) * 3 * d), *xl2 = malloc(sizeof(double) * d);
    embed(m, token, x, t3);
    for (int l = 0; l < m->L; ++l) {
        double *sa = s->shift_att + (size_t)l * d;
        tmix_front(m, l, x, sa, v_first, &w);
        memcpy(sa, w.xl, sizeof(double) * d);
        for (int h = 0; h < H; ++h) {
            double *S = s->wkv + ((size_t)l * H + h) * N * N;
            orc_wkv_step(N, S, w.r + h * N, w.decay + h * N, w.kh + h * N, w.a + h * N,
                         w.kp + h * N, w.vp + h * N, w.y + h * N);
        }
        tmix_back(m, l, x, &w);
        double *sf = s->shift_ffn + (size_t)l * d;
        cmix(m, l, x, sf, xl2, &w);
        memcpy(sf, xl2, sizeof(double) * d);
    }
    if (logits) head(m, x, logits, t3);
    free(pool); free(x); free(v_first); free(t3); free(xl2);
    return 0;
}

/*
 * Chunked prefill of T tokens of one sequence, layer-major: every layer runs
 * over the whole block before the next, the token-shift inputs come from a
 * shifted copy of the block, and the state update of each block of `chunk`
 * tokens uses orc_wkv_chunk.  logits_all ([T][V]) may be NULL; if not, the
 * logits after every token are written.
 */
int orc_prefill_chunked(const orc_model *m, orc_state *s, const int32_t *tokens, int T,
                        int chunk, double *logits_all) {
    if (T <= 0 || chunk <= 0) return -1;
    for (int t = 0; t < T; ++t)
        if (tokens[t] < 0 || tokens[t] >= m->V) return -1;
    int d = m->d, N = m->N, H = m->H;
    size_t Td = (size_t)T * d;
    double *X = malloc(sizeof(double) * Td);      /* residual stream, [T][d] */
    double *VF = malloc(sizeof(double) * Td);     /* layer-0 values */
    double *XL = malloc(sizeof(double) * Td);     /* LayerNorm outputs of the block */
    double *PREV = malloc(sizeof(double) * Td);   /* shifted copy */
    /* per-token time-mix quantities kept across the block */
    double *R = malloc(sizeof(double) * Td), *DEC = malloc(sizeof(double) * Td);
    double *KH = malloc(sizeof(double) * Td), *AA = malloc(sizeof(double) * Td);
    double *KP = malloc(sizeof(double) * Td), *VP = malloc(sizeof(double) * Td);
    double *G = malloc(sizeof(double) * Td), *Y = malloc(sizeof(double) * Td);
    double *hr = malloc(sizeof(double) * T * N), *hd = malloc(sizeof(double) * T * N);
    double *hk = malloc(sizeof(double) * T * N), *ha = malloc(sizeof(double) * T * N);
    double *hp = malloc(sizeof(double) * T * N), *hv = malloc(sizeof(double) * T * N);
    double *hy = malloc(sizeof(double) * T * N);
    double *t3 = malloc(sizeof(double) * 3 * d);
    orc_tok w;
    double *pool = tok_alloc(m, &w);
    for (int t = 0; t < T; ++t) embed(m, tokens[t], X + (size_t)t * d, t3);
    for (int l = 0; l < m->L; ++l) {
        double *sa = s->shift_att + (size_t)l * d;
        /* LayerNorm outputs of the whole block first, so that the shifted copy exists */
        {
            double *gam = t3, *bet = t3 + d;
            vec16(d, LT(m, l, T_LN1W), gam);
            vec16(d, LT(m, l, T_LN1B), bet);
            for (int t = 0; t < T; ++t)
                orc_layernorm(d, X + (size_t)t * d, gam, bet, 1e-5, XL + (size_t)t * d);
            memcpy(PREV, sa, sizeof(double) * d);
            memcpy(PREV + d, XL, sizeof(double) * (Td - d));
            memcpy(sa, XL + Td - d, sizeof(double) * d);
        }
        for (int t = 0; t < T; ++t) {
            tmix_front(m, l, X + (size_t)t * d, PREV + (size_t)t * d, VF + (size_t)t * d, &w);
            memcpy(R + (size_t)t * d, w.r, sizeof(double) * d);
            memcpy(DEC + (size_t)t * d, w.decay, sizeof(double) * d);
            memcpy(KH + (size_t)t * d, w.kh, sizeof(double) * d);
            memcpy(AA + (size_t)t * d, w.a, sizeof(double) * d);
            memcpy(KP + (size_t)t * d, w.kp, sizeof(double) * d);
            memcpy(VP + (size_t)t * d, w.vp, sizeof(double) * d);
            memcpy(G + (size_t)t * d, w.g, sizeof(double) * d);
        }
        for (int h = 0; h < H; ++h) {
            double *S = s->wkv + ((size_t)l * H + h) * N * N;
            for (int t = 0; t < T; ++t) {
                size_t o = (size_t)t * d + (size_t)h * N;
                memcpy(hr + t * N, R + o, sizeof(double) * N);
                memcpy(hd + t * N, DEC + o, sizeof(double) * N);
                memcpy(hk + t * N, KH + o, sizeof(double) * N);
                memcpy(ha + t * N, AA + o, sizeof(double) * N);
                memcpy(hp + t * N, KP + o, sizeof(double) * N);
                memcpy(hv + t * N, VP + o, sizeof(double) * N);
            }
            for (int t0 = 0; t0 < T; t0 += chunk) {
                int c = T - t0 < chunk ? T - t0 : chunk;
                orc_wkv_chunk(N, c, S, hr + t0 * N, hd + t0 * N, hk + t0 * N, ha + t0 * N,
                              hp + t0 * N, hv + t0 * N, hy + t0 * N);
            }
            for (int t = 0; t < T; ++t)
                memcpy(Y + (size_t)t * d + (size_t)h * N, hy + t * N, sizeof(double) * N);
        }
        for (int t = 0; t < T; ++t) {
            memcpy(w.y, Y + (size_t)t * d, sizeof(double) * d);
            memcpy(w.r, R + (size_t)t * d, sizeof(double) * d);
            memcpy(w.kp, KP + (size_t)t * d, sizeof(double) * d);
            memcpy(w.vp, VP + (size_t)t * d, sizeof(double) * d);
            memcpy(w.g, G + (size_t)t * d, sizeof(double) * d);
            tmix_back(m, l, X + (size_t)t * d, &w);
        }
        /* channel mix over the block */
        double *sf = s->shift_ffn + (size_t)l * d;
        {
            double *gam = t3, *bet = t3 + d;
            vec16(d, LT(m, l, T_LN2W), gam);
            vec16(d, LT(m, l, T_LN2B), bet);
            for (int t = 0; t < T; ++t)
                orc_layernorm(d, X + (size_t)t * d, gam, bet, 1e-5, XL + (size_t)t * d);
            memcpy(PREV, sf, sizeof(double) * d);
            memcpy(PREV + d, XL, sizeof(double) * (Td - d));
            memcpy(sf, XL + Td - d, sizeof(double) * d);
        }
        double *scratch = malloc(sizeof(double) * d);
        for (int t = 0; t < T; ++t) cmix(m, l, X + (size_t)t * d, PREV + (size_t)t * d, scratch, &w);
        free(scratch);
    }
    if (logits_all)
        for (int t = 0; t < T; ++t) head(m, X + (size_t)t * d, logits_all + (size_t)t * m->V, t3);
    free(X); free(VF); free(XL); free(PREV); free(R); free(DEC); free(KH); free(AA);
    free(KP); free(VP); free(G); free(Y); free(hr); free(hd); free(hk); free(ha); free(hp);
    free(hv); free(hy); free(t3); free(pool);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Sampler.                                                                   */
/* ------------------------------------------------------------------------- */

/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): 10 rounds of the 4x32 round
 * function with multipliers 0xD2511F53 / 0xCD9E8D57 and Weyl key increments
 * 0x9E3779B9 / 0xBB67AE85. */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0, n1 = lo1, n2 = hi0 ^ c3 ^ k1, n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* 64-bit uniform draw number `n` of the stream keyed by `seed`. */
uint64_t orc_draw_u64(uint64_t seed, uint64_t n) {
    uint32_t ctr[4] = {(uint32_t)n, (uint32_t)(n >> 32), 0u, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t o[4];
    orc_philox4x32_10(ctr, key, o);
    return (uint64_t)o[0] | ((uint64_t)o[1] << 32);
}

/*
 * 2^e for e <= 0 in fp32: Cody-Waite split e = n + f with n = nearest integer
 * (f in [-1/2, 1/2], exact), 2^f from its Taylor series in f*ln2 to degree 7
 * (truncation error < 6e-9, below fp32 resolution), evaluated by Horner with
 * fused multiply-adds, then scaled by the exact power 2^n.  Coefficients are
 * (ln 2)^k / k! rounded to fp32.
 */
static const float EXP2_C[8] = {
    1.0f, 0.693147180559945309f, 0.240226506959100712f, 0.0555041086648215800f,
    0.00961812910762847717f, 0.00133335581464284434f, 0.000154035303933816099f,
    0.0000152527338040598403f};

float orc_exp2(float e) {
    if (!(e > -126.0f)) return 0.0f;
    if (e > 0.0f) e = 0.0f;
    float n = floorf(e + 0.5f);
    float f = e - n;
    float p = EXP2_C[7];
    for (int k = 6; k >= 0; --k) p = fmaf(p, f, EXP2_C[k]);
    union { uint32_t u; float f; } sc;
    sc.u = (uint32_t)((int)n + 127) << 23;
    return p * sc.f;
}

typedef struct {
    float temperature, top_p;
    int32_t top_k;
    float presence, frequency, penalty_decay;
    uint64_t seed;
    int32_t greedy;
} orc_sampling;

static const float ORC_LOG2E = 1.44269504088896340736f;

/* integer weight 2^24 * 2^((l - m) * log2(e) / T), floor */
static uint32_t qweight(float l, float m, float T) {
    float dlt = l - m;
    if (T != 1.0f) dlt = dlt / T;
    float e = dlt * ORC_LOG2E;
    float p = orc_exp2(e);
    return (uint32_t)floorf(p * 16777216.0f);
}

static const uint32_t *g_sort_q;
static int cmp_desc(const void *pa, const void *pb) {
    int a = *(const int *)pa, b = *(const int *)pb;
    if (g_sort_q[a] != g_sort_q[b]) return g_sort_q[a] > g_sort_q[b] ? -1 : 1;
    return a < b ? -1 : (a > b);
}

/*
 * Integer sampling weights and the kept set for one row of fp32 logits [V]:
 *   1. penalty: l_i = logit_i - ((occ_i > 0 ? presence : 0) + occ_i * frequency)
 *   2. q1_i = floor(2^24 * 2^((l_i - max l) log2 e))
 *   3. top-p keeps every i with q1_i >= tp, tp the largest value whose tail mass
 *      sum_{q1_j >= tp} q1_j reaches ceil(top_p * sum q1) (at least 1); ties at
 *      the cut value are all kept
 *   4. top-k (k > 0) keeps the first k in the order (q1 desc, index asc)
 *   5. over the kept set, qT_i = floor(2^24 * 2^((l_i - max l)/T log2 e)); 0 elsewhere
 * q1, qT, keep are caller arrays of V words; scratch holds 2*V words.
 * Not reentrant (the sort comparator reads a file-scope pointer).
 */
void orc_sample_weights(int V, const float *logits, const float *occ, const orc_sampling *p,
                        uint32_t *q1, uint32_t *qT, uint32_t *keep, uint32_t *scratch) {
    float *l = (float *)scratch;
    int *order = (int *)(scratch + V);
    for (int i = 0; i < V; ++i) {
        float o = occ[i];
        float pres = o > 0.0f ? p->presence : 0.0f;
        float t = o * p->frequency;
        t = pres + t;
        l[i] = logits[i] - t;
    }
    float mx = l[0];
    for (int i = 1; i < V; ++i)
        if (l[i] > mx) mx = l[i];
    uint64_t Q1 = 0;
    for (int i = 0; i < V; ++i) {
        q1[i] = qweight(l[i], mx, 1.0f);
        Q1 += q1[i];
    }
    uint64_t target = (uint64_t)ceil((double)p->top_p * (double)Q1);
    if (target < 1) target = 1;
    if (target > Q1) target = Q1;
    for (int i = 0; i < V; ++i) order[i] = i;
    g_sort_q = q1;
    qsort(order, (size_t)V, sizeof(int), cmp_desc);
    uint64_t acc = 0;
    uint32_t tp = 0;
    for (int r = 0; r < V; ++r) {
        acc += q1[order[r]];
        if (acc >= target) {
            tp = q1[order[r]];
            break;
        }
    }
    for (int i = 0; i < V; ++i) keep[i] = q1[i] >= tp;
    if (p->top_k > 0 && p->top_k < V)
        for (int r = p->top_k; r < V; ++r) keep[order[r]] = 0;
    for (int i = 0; i < V; ++i)
        qT[i] = !keep[i] ? 0u : (p->temperature == 1.0f ? q1[i] : qweight(l[i], mx, p->temperature));
}

/* The first index i (ascending) whose running sum of w exceeds r, for r in [0, sum w). */
int32_t orc_pick(int V, const uint32_t *w, uint64_t r) {
    uint64_t acc = 0;
    for (int i = 0; i < V; ++i) {
        acc += w[i];
        if (acc > r) return i;
    }
    return -1;
}

/*
 * Sample one token from fp32 logits [V].
 *  greedy (or temperature <= 0): argmax of the raw logits, lowest index on ties;
 *    occurrence counts are neither read nor written.
 *  otherwise: weights and kept set as in orc_sample_weights, then
 *    r = floor(u * R / 2^64) with u the Philox draw number `draw_index` of the
 *    stream keyed by the seed and R = sum qT; token = orc_pick(qT, r); finally
 *    occ_i *= penalty_decay for all i and occ[token] += 1.
 * scratch: 5*V words.  kept_out: V words (kept-set flags).
 */
int32_t orc_sample(int V, const float *logits, float *occ, const orc_sampling *p,
                   uint64_t draw_index, uint32_t *scratch, uint32_t *kept_out) {
    if (p->greedy || !(p->temperature > 0.0f)) {
        int best = 0;
        for (int i = 1; i < V; ++i)
            if (logits[i] > logits[best]) best = i;
        for (int i = 0; i < V; ++i) kept_out[i] = (i == best);
        return best;
    }
    uint32_t *q1 = scratch, *qT = scratch + V, *rest = scratch + 2 * (size_t)V;
    orc_sample_weights(V, logits, occ, p, q1, qT, kept_out, rest);
    uint64_t R = 0;
    for (int i = 0; i < V; ++i) R += qT[i];
    uint64_t u = orc_draw_u64(p->seed, draw_index);
    uint64_t rr = (uint64_t)(((unsigned __int128)u * (unsigned __int128)R) >> 64);
    int32_t tok = orc_pick(V, qT, rr);
    for (int i = 0; i < V; ++i) occ[i] = occ[i] * p->penalty_decay;
    occ[tok] = occ[tok] + 1.0f;
    return tok;
}
