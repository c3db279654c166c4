/*
 * oracle.c — fp64 CPU oracle of one batch-1 Llama-style decode step.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h): used by tests/, the package smoke
 * check and the benchmark's CPU-baseline leg, never by the product path.
 *
 * Source of truth: "Revolution der KI-Beschleunigung: Wie ein Low-Latency
 * Megakernel den Llama-1B Turbo zündet" (dasgeld.co). The article describes a
 * single-kernel bf16 decode forward pass of Llama-1B at batch 1 and states
 * the speed-up costs no accuracy, so the result to reproduce is the plain
 * Llama decode step. The article leaves every formula open; the readings
 * taken (pre-norm RMSNorm with eps inside the root, rotate-half RoPE without
 * frequency scaling, causal attention including the current token, scale
 * 1/sqrt(hd), contiguous GQA groups, tied unscaled embedding, no biases,
 * bf16 post-RoPE KV cache, lowest-index argmax) are the standard Llama ones.
 *
 * Plain sequential loops in double. The only parallelism is an OpenMP
 * split over independent output rows / heads, which changes no arithmetic.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int g_threads = 0;

void orc_set_threads(int n) { g_threads = n; }

int orc_get_threads(void) {
#ifdef _OPENMP
    return g_threads > 0 ? g_threads : omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- bf16 <-> double ---------------------------------------------------- */

double orc_bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16; /* bf16 is the top half of an IEEE binary32 */
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

uint16_t orc_f64_to_bf16(double x) {
    /* bf16: 1 sign, 8 exponent, 7 fraction bits (8 significant bits). Round
     * |x| to the nearest multiple of the bf16 quantum at its binade, ties to
     * even (nearbyint in the default rounding mode), then re-encode exactly. */
    if (isnan(x)) return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0) return sign;
    if (isinf(a)) return sign | 0x7F80;
    int e;
    frexp(a, &e);                           /* a = m * 2^e, m in [0.5, 1) */
    int qexp = (e - 1 >= -126) ? e - 8 : -133; /* quantum: normal / subnormal */
    double r = nearbyint(ldexp(a, -qexp));   /* exact scaling by a power of two */
    r = ldexp(r, qexp);
    if (r >= ldexp(1.0, 128)) return sign | 0x7F80; /* overflow to infinity */
    float f = (float)r; /* exactly representable: at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

/* ---- primitives --------------------------------------------------------- */

void orc_rmsnorm(const double *x, const uint16_t *g, int n, double eps, double *out) {
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss / (double)n + eps);
    for (int i = 0; i < n; ++i) out[i] = x[i] * inv * orc_bf16_to_f64(g[i]);
}

void orc_matvec(const uint16_t *W, int64_t rows, int64_t cols, const double *x, double *y) {
    int nt = orc_get_threads();
    (void)nt;
#pragma omp parallel for schedule(static) num_threads(nt)
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t *row = W + r * cols;
        double acc = 0.0;
        for (int64_t c = 0; c < cols; ++c) acc += orc_bf16_to_f64(row[c]) * x[c];
        y[r] = acc;
    }
}

void orc_rope(double *v, int hd, int64_t pos, double theta) {
    int half = hd / 2;
    for (int i = 0; i < half; ++i) {
        double freq = pow(theta, -2.0 * (double)i / (double)hd);
        double ang = (double)pos * freq;
        double c = cos(ang), s = sin(ang);
        double a = v[i], b = v[i + half];
        v[i] = a * c - b * s;
        v[i + half] = b * c + a * s;
    }
}

double orc_silu(double z) { return z / (1.0 + exp(-z)); }

void orc_softmax(const double *s, int n, double *p) {
    double m = -INFINITY;
    for (int j = 0; j < n; ++j)
        if (s[j] > m) m = s[j];
    double sum = 0.0;
    for (int j = 0; j < n; ++j) {
        p[j] = exp(s[j] - m);
        sum += p[j];
    }
    for (int j = 0; j < n; ++j) p[j] /= sum;
}

void orc_attend(const double *q, const uint16_t *K, const uint16_t *V, int T, int hd, double *o) {
    double *s = (double *)calloc((size_t)(T > 0 ? T : 1), sizeof(double));
    double *p = (double *)calloc((size_t)(T > 0 ? T : 1), sizeof(double));
    double scale = 1.0 / sqrt((double)hd);
    for (int j = 0; j < T; ++j) {
        double dot = 0.0;
        for (int i = 0; i < hd; ++i) dot += q[i] * orc_bf16_to_f64(K[(int64_t)j * hd + i]);
        s[j] = dot * scale;
    }
    orc_softmax(s, T, p);
    for (int i = 0; i < hd; ++i) o[i] = 0.0;
    for (int j = 0; j < T; ++j)
        for (int i = 0; i < hd; ++i) o[i] += p[j] * orc_bf16_to_f64(V[(int64_t)j * hd + i]);
    free(s);
    free(p);
}

int orc_argmax(const double *v, int n) {
    int best = 0;
    for (int i = 1; i < n; ++i)
        if (v[i] > v[best]) best = i; /* strict: keeps the lowest index on ties */
    return best;
}

static int valid_config(const orc_config *c) {
    return c && c->n_layers > 0 && c->d_model > 0 && c->n_heads > 0 && c->n_kv_heads > 0 &&
           c->head_dim > 0 && (c->head_dim % 2) == 0 && c->ffn_dim > 0 && c->vocab > 0 &&
           (c->n_heads % c->n_kv_heads) == 0;
}

/* Final norm + tied LM head + greedy argmax. */
static int lm_head(const orc_config *c, const orc_weights *w, const double *x, double *logits) {
    int d = c->d_model;
    double *xh = (double *)malloc(sizeof(double) * (size_t)d);
    orc_rmsnorm(x, w->final_norm, d, c->rms_eps, xh);
    orc_matvec(w->embed, c->vocab, d, xh, logits);
    free(xh);
    return orc_argmax(logits, c->vocab);
}


/* x += Wd (silu(Wg xh) * (Wu xh)),  xh = RMSNorm(x) * g_mlp  (in place). */
void orc_mlp_block(const orc_layer *L, int d, int F, double eps, double *x) {
    double *xh = (double *)malloc(sizeof(double) * (size_t)d);
    double *gt = (double *)malloc(sizeof(double) * (size_t)F);
    double *up = (double *)malloc(sizeof(double) * (size_t)F);
    double *t = (double *)malloc(sizeof(double) * (size_t)d);
    orc_rmsnorm(x, L->mlp_norm, d, eps, xh);
    orc_matvec(L->w_gate, F, d, xh, gt);
    orc_matvec(L->w_up, F, d, xh, up);
    for (int i = 0; i < F; ++i) gt[i] = orc_silu(gt[i]) * up[i];
    orc_matvec(L->w_down, d, F, gt, t);
    for (int i = 0; i < d; ++i) x[i] += t[i];
    free(xh); free(gt); free(up); free(t);
}

/* ---- one decode step (incremental, with the KV cache) ------------------ */

int orc_decode_step(const orc_config *c, const orc_weights *w, const orc_kv *kv, int token,
                    int pos, double *logits) {
    if (!valid_config(c) || !w || !kv || !logits) return -1;
    if (token < 0 || token >= c->vocab || pos < 0 || pos >= kv->max_seq) return -1;
    const int d = c->d_model, H = c->n_heads, Hkv = c->n_kv_heads, hd = c->head_dim;
    const int F = c->ffn_dim, G = H / Hkv, S = kv->max_seq;

    double *x = (double *)malloc(sizeof(double) * (size_t)d);
    double *xh = (double *)malloc(sizeof(double) * (size_t)d);
    double *q = (double *)malloc(sizeof(double) * (size_t)H * hd);
    double *k = (double *)malloc(sizeof(double) * (size_t)Hkv * hd);
    double *v = (double *)malloc(sizeof(double) * (size_t)Hkv * hd);
    double *o = (double *)malloc(sizeof(double) * (size_t)H * hd);
    double *t = (double *)malloc(sizeof(double) * (size_t)d);

    for (int i = 0; i < d; ++i) x[i] = orc_bf16_to_f64(w->embed[(int64_t)token * d + i]);

    for (int l = 0; l < c->n_layers; ++l) {
        const orc_layer *L = &w->layers[l];
        uint16_t *Kl = kv->k + (int64_t)l * kv->layer_stride;
        uint16_t *Vl = kv->v + (int64_t)l * kv->layer_stride;

        orc_rmsnorm(x, L->attn_norm, d, c->rms_eps, xh);
        orc_matvec(L->wq, (int64_t)H * hd, d, xh, q);
        orc_matvec(L->wk, (int64_t)Hkv * hd, d, xh, k);
        orc_matvec(L->wv, (int64_t)Hkv * hd, d, xh, v);
        for (int h = 0; h < H; ++h) orc_rope(q + (int64_t)h * hd, hd, pos, c->rope_theta);
        for (int h = 0; h < Hkv; ++h) orc_rope(k + (int64_t)h * hd, hd, pos, c->rope_theta);

        /* KV append: bf16 rows at `pos`. */
        for (int h = 0; h < Hkv; ++h)
            for (int i = 0; i < hd; ++i) {
                int64_t off = ((int64_t)h * S + pos) * hd + i;
                Kl[off] = orc_f64_to_bf16(k[(int64_t)h * hd + i]);
                Vl[off] = orc_f64_to_bf16(v[(int64_t)h * hd + i]);
            }

        /* Causal GQA attention over positions 0..pos of kv head h / G. */
        for (int h = 0; h < H; ++h) {
            int kvh = h / G;
            orc_attend(q + (int64_t)h * hd, Kl + (int64_t)kvh * S * hd, Vl + (int64_t)kvh * S * hd,
                       pos + 1, hd, o + (int64_t)h * hd);
        }

        orc_matvec(L->wo, d, (int64_t)H * hd, o, t);
        for (int i = 0; i < d; ++i) x[i] += t[i];

        orc_mlp_block(L, d, F, c->rms_eps, x);
    }
    int tok = lm_head(c, w, x, logits);
    free(x); free(xh); free(q); free(k); free(v); free(o); free(t);
    return tok;
}

/* ---- full causal forward (no incremental cache reuse) ------------------ */

int orc_full_forward(const orc_config *c, const orc_weights *w, const int *tokens, int n,
                     double *logits) {
    if (!valid_config(c) || !w || !tokens || n <= 0 || !logits) return -1;
    const int d = c->d_model, H = c->n_heads, Hkv = c->n_kv_heads, hd = c->head_dim;
    const int F = c->ffn_dim, G = H / Hkv;
    for (int i = 0; i < n; ++i)
        if (tokens[i] < 0 || tokens[i] >= c->vocab) return -1;

    /* Hidden states of all positions, layer by layer. */
    double *X = (double *)malloc(sizeof(double) * (size_t)n * d);
    double *xh = (double *)malloc(sizeof(double) * (size_t)d);
    double *Q = (double *)malloc(sizeof(double) * (size_t)n * H * hd);
    double *kk = (double *)malloc(sizeof(double) * (size_t)Hkv * hd);
    double *vv = (double *)malloc(sizeof(double) * (size_t)Hkv * hd);
    /* Per kv head, rows of all positions: [Hkv][n][hd] bf16. */
    uint16_t *Kb = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)Hkv * n * hd);
    uint16_t *Vb = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)Hkv * n * hd);
    double *o = (double *)malloc(sizeof(double) * (size_t)H * hd);
    double *t = (double *)malloc(sizeof(double) * (size_t)d);

    for (int p = 0; p < n; ++p)
        for (int i = 0; i < d; ++i) X[(int64_t)p * d + i] = orc_bf16_to_f64(w->embed[(int64_t)tokens[p] * d + i]);

    for (int l = 0; l < c->n_layers; ++l) {
        const orc_layer *L = &w->layers[l];
        /* Projections of every position first. */
        for (int p = 0; p < n; ++p) {
            orc_rmsnorm(X + (int64_t)p * d, L->attn_norm, d, c->rms_eps, xh);
            double *qp = Q + (int64_t)p * H * hd;
            orc_matvec(L->wq, (int64_t)H * hd, d, xh, qp);
            orc_matvec(L->wk, (int64_t)Hkv * hd, d, xh, kk);
            orc_matvec(L->wv, (int64_t)Hkv * hd, d, xh, vv);
            for (int h = 0; h < H; ++h) orc_rope(qp + (int64_t)h * hd, hd, p, c->rope_theta);
            for (int h = 0; h < Hkv; ++h) {
                orc_rope(kk + (int64_t)h * hd, hd, p, c->rope_theta);
                for (int i = 0; i < hd; ++i) {
                    Kb[((int64_t)h * n + p) * hd + i] = orc_f64_to_bf16(kk[(int64_t)h * hd + i]);
                    Vb[((int64_t)h * n + p) * hd + i] = orc_f64_to_bf16(vv[(int64_t)h * hd + i]);
                }
            }
        }
        /* Then causal attention and the MLP of every position. */
        for (int p = 0; p < n; ++p) {
            double *x = X + (int64_t)p * d;
            for (int h = 0; h < H; ++h)
                orc_attend(Q + ((int64_t)p * H + h) * hd, Kb + (int64_t)(h / G) * n * hd,
                           Vb + (int64_t)(h / G) * n * hd, p + 1, hd, o + (int64_t)h * hd);
            orc_matvec(L->wo, d, (int64_t)H * hd, o, t);
            for (int i = 0; i < d; ++i) x[i] += t[i];
            orc_mlp_block(L, d, F, c->rms_eps, x);
        }
    }
    int tok = lm_head(c, w, X + (int64_t)(n - 1) * d, logits);
    free(X); free(xh); free(Q); free(kk); free(vv); free(Kb); free(Vb);
    free(o); free(t);
    return tok;
}

/* ---- W2A8 projections (see oracle.h) ----------------------------------- */

float orc_w2a8_quantize(const double *x, int n, int8_t *codes) {
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        const float a = fabsf((float)x[i]);
        if (a > amax) amax = a;
    }
    const float s = 127.0f / (amax > 1e-5f ? amax : 1e-5f);
    for (int i = 0; i < n; ++i) {
        const float v = rintf((float)x[i] * s);
        codes[i] = (int8_t)(v < -128.0f ? -128.0f : (v > 127.0f ? 127.0f : v));
    }
    return s;
}

void orc_matvec_w2a8(const int8_t *Wq, float beta, int64_t rows, int64_t cols, const double *x, double *y) {
    int8_t *q = (int8_t *)malloc((size_t)cols);
    const float s = orc_w2a8_quantize(x, (int)cols, q);
    const double f = (double)beta / (double)s;
#pragma omp parallel for schedule(static) num_threads(orc_get_threads())
    for (int64_t r = 0; r < rows; ++r) {
        int64_t acc = 0;
        for (int64_t c = 0; c < cols; ++c) acc += (int64_t)Wq[r * cols + c] * (int64_t)q[c];
        y[r] = f * (double)acc;
    }
    free(q);
}

int orc_decode_step_w2a8(const orc_config *c, const orc_weights_w2 *w, const orc_kv *kv, int token,
                         int pos, double *logits) {
    if (!valid_config(c) || !w || !kv || !logits) return -1;
    if (token < 0 || token >= c->vocab || pos < 0 || pos >= kv->max_seq) return -1;
    const int d = c->d_model, H = c->n_heads, Hkv = c->n_kv_heads, hd = c->head_dim;
    const int F = c->ffn_dim, G = H / Hkv, S = kv->max_seq;

    double *x = (double *)malloc(sizeof(double) * (size_t)d);
    double *xh = (double *)malloc(sizeof(double) * (size_t)d);
    double *q = (double *)malloc(sizeof(double) * (size_t)H * hd);
    double *k = (double *)malloc(sizeof(double) * (size_t)Hkv * hd);
    double *v = (double *)malloc(sizeof(double) * (size_t)Hkv * hd);
    double *o = (double *)malloc(sizeof(double) * (size_t)H * hd);
    double *t = (double *)malloc(sizeof(double) * (size_t)d);
    double *gt = (double *)malloc(sizeof(double) * (size_t)F);
    double *up = (double *)malloc(sizeof(double) * (size_t)F);

    for (int i = 0; i < d; ++i) x[i] = orc_bf16_to_f64(w->embed[(int64_t)token * d + i]);

    for (int l = 0; l < c->n_layers; ++l) {
        const orc_layer_w2 *L = &w->layers[l];
        uint16_t *Kl = kv->k + (int64_t)l * kv->layer_stride;
        uint16_t *Vl = kv->v + (int64_t)l * kv->layer_stride;

        orc_rmsnorm(x, L->attn_norm, d, c->rms_eps, xh);
        orc_matvec_w2a8(L->wq, L->beta_q, (int64_t)H * hd, d, xh, q);
        orc_matvec_w2a8(L->wk, L->beta_k, (int64_t)Hkv * hd, d, xh, k);
        orc_matvec_w2a8(L->wv, L->beta_v, (int64_t)Hkv * hd, d, xh, v);
        for (int h = 0; h < H; ++h) orc_rope(q + (int64_t)h * hd, hd, pos, c->rope_theta);
        for (int h = 0; h < Hkv; ++h) orc_rope(k + (int64_t)h * hd, hd, pos, c->rope_theta);
        for (int h = 0; h < Hkv; ++h)
            for (int i = 0; i < hd; ++i) {
                int64_t off = ((int64_t)h * S + pos) * hd + i;
                Kl[off] = orc_f64_to_bf16(k[(int64_t)h * hd + i]);
                Vl[off] = orc_f64_to_bf16(v[(int64_t)h * hd + i]);
            }
        for (int h = 0; h < H; ++h) {
            int kvh = h / G;
            orc_attend(q + (int64_t)h * hd, Kl + (int64_t)kvh * S * hd, Vl + (int64_t)kvh * S * hd,
                       pos + 1, hd, o + (int64_t)h * hd);
        }
        orc_matvec_w2a8(L->wo, L->beta_o, d, (int64_t)H * hd, o, t);
        for (int i = 0; i < d; ++i) x[i] += t[i];

        orc_rmsnorm(x, L->mlp_norm, d, c->rms_eps, xh);
        orc_matvec_w2a8(L->w_gate, L->beta_gate, F, d, xh, gt);
        orc_matvec_w2a8(L->w_up, L->beta_up, F, d, xh, up);
        for (int i = 0; i < F; ++i) gt[i] = orc_silu(gt[i]) * up[i];
        orc_matvec_w2a8(L->w_down, L->beta_down, d, F, gt, t);
        for (int i = 0; i < d; ++i) x[i] += t[i];
    }
    const orc_weights head = {w->embed, w->final_norm, NULL};  /* the LM head stays bf16 */
    int tok = lm_head(c, &head, x, logits);
    free(x); free(xh); free(q); free(k); free(v); free(o); free(t); free(gt); free(up);
    return tok;
}
