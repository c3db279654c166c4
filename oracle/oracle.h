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

/* ---- W2A8 projections -------------------------------------------------
 * Ternary weights and 8-bit activations, as the page "BitNet 1.58bit GPU
 * Inference Kernel: Revolutionäre Effizienz für KI-Modelle mit
 * W2A8-Quantisierung" (dasgeld.co) describes its GEMV: 2-bit weights, 8-bit
 * activations, an integer dot product (dp4a). The page gives no formulas;
 * the plainest reading is BitNet b1.58's (Ma et al., 2024): a weight matrix
 * is beta * Wq with Wq in {-1, 0, +1} and one fp32 scale beta per matrix; an
 * input vector x is quantised per token by its absolute maximum,
 *     s = 127 / max(max_i |x_i|, 1e-5),   x_q[i] = clamp(rint(x_i * s), -128, 127),
 * in fp32 arithmetic (x first rounded to fp32: the decision is taken in the
 * kernel's precision), and
 *     y[r] = (beta / s) * sum_c Wq[r][c] * x_q[c]   (exact integer sum).  */

/* Activation codes of x[n]; returns the scale s. */
float orc_w2a8_quantize(const double *x, int n, int8_t *codes);

/* y[r] = beta / s * sum_c Wq[r][c] x_q[c] for Wq int8 row-major [rows][cols]. */
void orc_matvec_w2a8(const int8_t *Wq, float beta, int64_t rows, int64_t cols, const double *x, double *y);

/* A layer whose seven projections are W2A8 (norm gains stay bf16). */
typedef struct {
    const uint16_t *attn_norm, *mlp_norm;
    const int8_t *wq, *wk, *wv, *wo, *w_gate, *w_up, *w_down;
    float beta_q, beta_k, beta_v, beta_o, beta_gate, beta_up, beta_down;
} orc_layer_w2;

/* embed (bf16, also the tied LM head, which stays bf16) and final_norm as in
 * orc_weights; layers: [n_layers] W2A8 layers. */
typedef struct {
    const uint16_t *embed;
    const uint16_t *final_norm;
    const orc_layer_w2 *layers;
} orc_weights_w2;

/* orc_decode_step with every projection of every layer W2A8: the same step
 * with orc_matvec_w2a8 in place of orc_matvec for Wq, Wk, Wv, Wo, Wg, Wu,
 * Wd (each quantising its own input vector). Returns the greedy token, -1 on
 * bad arguments. */
int orc_decode_step_w2a8(const orc_config *cfg, const orc_weights_w2 *w, const orc_kv *kv, int token,
                         int pos, double *logits);

#ifdef __cplusplus
}
#endif
#endif
