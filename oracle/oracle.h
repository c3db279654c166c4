/*
 * oracle.h — plain, slow, obviously-correct CPU forward pass of one batch-1
 * Llama-style decode step, in fp64.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may include, link,
 * load or call this code: only the test suite, the package smoke check and
 * the CPU-baseline leg of the benchmark use it. It shares no code, header,
 * table or constant with the CUDA implementation.
 *
 * What it computes follows "Revolution der KI-Beschleunigung: Wie ein
 * Low-Latency Megakernel den Llama-1B Turbo zündet" (dasgeld.co), which
 * describes a fused batch-1 bf16 decode forward pass of Llama-1B and claims
 * no accuracy compromise (section on chat systems). The megakernel therefore
 * has to reproduce the standard Llama decode step, which is written out here
 * step by step:
 *
 *   x  = E[token]                                   (embedding, tied, unscaled)
 *   per layer:
 *     xh = x / sqrt(mean(x^2) + eps) * g_attn       (RMSNorm, pre-norm)
 *     q = Wq xh, k = Wk xh, v = Wv xh               (no biases)
 *     rotate q and k with RoPE at `pos` (pairs i, i+hd/2, freq theta^(-2i/hd))
 *     K[pos] = bf16(k), V[pos] = bf16(v)            (bf16 cache, post-RoPE keys)
 *     o_h = sum_j softmax_j(q_h . K_j / sqrt(hd)) V_j,  j = 0..pos, kv head = h / G
 *     x += Wo o
 *     xh = RMSNorm(x) * g_mlp
 *     x += Wd (silu(Wg xh) * (Wu xh))
 *   logits = E (RMSNorm(x) * g_final);  token = argmax (lowest index on ties)
 *
 * Weights, norm gains and the KV cache are bf16 (the article fixes bf16 as
 * the model precision); everything else is double. bf16 values are widened
 * exactly (bits << 16). Weight matrices are row-major [out][in].
 *
 * Parity pins: every function here is pinned by tests/test_oracle_pins.py
 * against closed forms, invariants, library routines (numpy float64) or a
 * separately coded full causal forward. End-to-end logits of random models
 * have no printed values on the pages, so beyond those pins the end-to-end
 * result is "parity unpinned" except through its pinned parts.
 */
#ifndef MK_ORACLE_H
#define MK_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int32_t n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn_dim, vocab;
    double rms_eps, rope_theta;
} orc_config;

typedef struct {
    const uint16_t *attn_norm, *wq, *wk, *wv, *wo, *mlp_norm, *w_gate, *w_up, *w_down;
} orc_layer;

typedef struct {
    const uint16_t *embed;      /* [vocab][d_model] */
    const uint16_t *final_norm; /* [d_model] */
    const orc_layer *layers;    /* [n_layers] */
} orc_weights;

/* KV cache view for one sequence: element (l, kvh, t, i) lives at
 * base + l*layer_stride + (kvh*max_seq + t)*head_dim + i.                 */
typedef struct {
    uint16_t *k, *v;
    int64_t layer_stride;
    int32_t max_seq;
} orc_kv;

/* bf16 <-> double. */
double   orc_bf16_to_f64(uint16_t b);
uint16_t orc_f64_to_bf16(double x); /* round to nearest, ties to even */

/* Number of OpenMP threads used by the parallel loops (0 = library default). */
void orc_set_threads(int n);
int  orc_get_threads(void);

/* out[i] = x[i] / sqrt(sum(x^2)/n + eps) * g[i] */
void orc_rmsnorm(const double *x, const uint16_t *g, int n, double eps, double *out);

/* y[r] = sum_c W[r][c] * x[c], W bf16 row-major [rows][cols] */
void orc_matvec(const uint16_t *W, int64_t rows, int64_t cols, const double *x, double *y);

/* In-place rotary embedding of one head vector v[hd] at position pos. */
void orc_rope(double *v, int hd, int64_t pos, double theta);

/* silu(z) = z / (1 + exp(-z)) */
double orc_silu(double z);

/* x += Wd (silu(Wg xh) * (Wu xh)) with xh = RMSNorm(x) * mlp_norm, in place. */
void orc_mlp_block(const orc_layer *L, int d, int F, double eps, double *x);

/* Softmax of s[n] into p[n] (max-subtracted). */
void orc_softmax(const double *s, int n, double *p);

/* One query head over T cached positions: o = sum_j softmax(q.K_j/sqrt(hd))_j V_j.
 * K and V point at [T][hd] bf16 rows (contiguous).                        */
void orc_attend(const double *q, const uint16_t *K, const uint16_t *V, int T, int hd, double *o);

/* Lowest index of the maximum. */
int orc_argmax(const double *v, int n);

/* One decode step: writes K/V at `pos` into the cache, fills logits[vocab],
 * returns the greedy token. Returns -1 on bad arguments.                   */
int orc_decode_step(const orc_config *cfg, const orc_weights *w, const orc_kv *kv,
                    int token, int pos, double *logits);

/* Separately coded full causal forward over tokens[0..n-1] starting at
 * position 0 with an empty cache: recomputes every position's keys and
 * values from scratch (rounded to bf16 like the cache format) and returns the
 * logits of the last position. Returns the greedy token, -1 on error.       */
int orc_full_forward(const orc_config *cfg, const orc_weights *w, const int *tokens, int n,
                     double *logits);

#ifdef __cplusplus
}
#endif
#endif
