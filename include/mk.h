/*
 * mk.h — C ABI of a persistent decode megakernel for Llama-style models on
 * one GB300 (sm_103a).
 *
 * What it implements: one batch-1 autoregressive decode step of a Llama-style
 * decoder (RMSNorm, QKV projection, RoPE, KV-cache append, grouped-query
 * attention, O-projection plus residual, SwiGLU MLP plus residual, final norm,
 * tied LM head, greedy argmax), fused into ONE persistent kernel launch, as
 * described in "Revolution der KI-Beschleunigung: Wie ein Low-Latency
 * Megakernel den Llama-1B Turbo zündet" (dasgeld.co):
 *   - all operations of the forward pass fused into a single kernel (the
 *     megakernel paragraphs);
 *   - a GPU interpreter that runs instruction sequences planned ahead on the
 *     host, one sequence per streaming multiprocessor, reused for every step
 *     without recompiling (the paragraph on the internal infrastructure);
 *   - dependencies resolved through counters in global memory, at the
 *     granularity of parts of a tensor (the synchronisation paragraph);
 *   - shared memory split into pages handed out to instructions so the next
 *     load starts while the current one finishes (the shared-memory
 *     paging paragraph);
 *   - bf16 model precision (the latency paragraph).
 * The glossary entry "Megakernel" (synthszr.com) describes the same design:
 * one launch working through a task list, counters and signals in memory.
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers unless a name says `host`.
 *   - bf16 tensors are row-major; matrices are [out_features][in_features].
 *   - Pointers handed to mk_create are borrowed: the caller owns them and
 *     must keep them alive and unmoved until mk_destroy. The library never
 *     writes the weights; of the KV cache it writes only row `position` of
 *     each layer of the stepping sequence's batch slot (slot 0 for the
 *     single-sequence calls).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls
 *     are asynchronous on it; a handle is not thread-safe and must not have
 *     two steps in flight on different streams at once.
 *   - Return value: MK_OK or a negative mk_status. The text of the last
 *     error on the calling thread is given by mk_last_error().
 */
#ifndef MK_H
#define MK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mk_status {
    MK_OK = 0,
    MK_ERR_INVALID_ARG = -1, /* null/misaligned pointer, bad size, token or position out of range */
    MK_ERR_CUDA = -2,        /* a CUDA runtime call failed (message in mk_last_error) */
    MK_ERR_LAUNCH = -3,      /* the persistent grid could not be made co-resident */
    MK_ERR_UNSUPPORTED = -4, /* device is not sm_103, or a shape the kernels do not handle */
    MK_ERR_TIMEOUT = -5,     /* a bounded wait inside the kernel expired (see mk_get_status) */
    MK_ERR_NOMEM = -6        /* device or host allocation failed */
} mk_status;

/* Model shape. Requirements: d_model and n_heads*head_dim are each one of
 * 256, 512, 768, 1024, 1536, 2048, 3072, 4096, and ffn_dim one of those or
 * 6144, 8192 (a row is split over 1, 2, 4 or 8 warps in slices of 256..1024); head_dim is 64 or 128; n_heads is a multiple of n_kv_heads, at
 * most 4 query heads per kv head; at most 127 layers. rms_eps is added to
 * the mean square inside the square root; rope_theta is the RoPE base. */
typedef struct mk_config {
    int32_t n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn_dim, vocab;
    int32_t max_seq;     /* positions in the KV cache per sequence */
    int32_t max_batch;   /* sequences in the KV cache (slot 0 for the single-sequence calls) */
    int32_t attn_splits; /* KV splits per kv head for attention, 0 = automatic */
    float rms_eps, rope_theta;
} mk_config;

/* bf16 device pointers of one layer: attn_norm [d], wq [n_heads*hd][d],
 * wk and wv [n_kv_heads*hd][d], wo [d][n_heads*hd], mlp_norm [d],
 * w_gate and w_up [ffn][d], w_down [d][ffn]. 16-byte aligned. */
typedef struct mk_layer_weights {
    const void *attn_norm, *wq, *wk, *wv, *wo, *mlp_norm, *w_gate, *w_up, *w_down;
} mk_layer_weights;

/* embed: bf16 [vocab][d], also the (tied) LM head. final_norm: bf16 [d].
 * layers: HOST array of n_layers entries (copied by mk_create). */
typedef struct mk_weights {
    const void *embed;
    const void *final_norm;
    const mk_layer_weights *layers;
} mk_weights;

/* bf16 device pointers, each [n_layers][max_batch][n_kv_heads][max_seq][head_dim].
 * Keys are stored after RoPE. */
typedef struct mk_kv_cache {
    void *k;
    void *v;
} mk_kv_cache;

typedef struct mk_handle mk_handle;

/* Plans the per-SM instruction queues for this model on the current device
 * (host scheduler), allocates the library's scratch (activations, attention
 * partials, dependency counters, queues, RoPE table) and uploads them.
 * With max_batch > 1, head_dim 64 and d_model a multiple of 64 it also plans
 * the fused batched step and keeps, for it, an fp16 copy of every layer
 * GEMV weight (2 bytes per weight, owned by the handle; exact for
 * magnitudes in fp16's normal range) and the LM head's scratch (its logits
 * and draw lists for max_batch sequences); if that does not fit, or a
 * weight lies beyond fp16's largest finite value (65504), batches run
 * sequence by sequence instead. Synchronous. On success *out receives
 * the handle.
 * Source: the article "Revolution der KI-Beschleunigung: Wie ein Low-Latency
 * Megakernel den Llama-1B Turbo zündet" (dasgeld.co), paragraph on the
 * internal infrastructure: a GPU interpreter runs
 * instruction sequences that are planned once on the host, one per SM, and
 * reused for many forward passes without recompiling. */
int mk_create(const mk_config *config, const mk_weights *weights, const mk_kv_cache *kv,
              mk_handle **out);

/* One decode step at `position` for token `token_id` (batch slot 0): writes
 * the new key/value row at `position`, attends over 0..position, and writes
 * the greedy next token to out_token (device int32[1]) and, if out_logits is
 * not NULL, the fp32 logits to out_logits (device float[vocab]).
 * Exactly one kernel launch.
 * Source: the same article, megakernel paragraphs (every step of the forward
 * pass fused into one kernel, no launch or teardown between steps) and
 * latency paragraph (one single-sequence forward pass in bf16). */
int mk_decode_step(mk_handle *h, int32_t token_id, int32_t position, float *out_logits,
                   int32_t *out_token, void *stream);

/* Same, with the token read from device memory (d_token_id, int32[1]) when
 * the step runs, so generation can chain out_token -> next step without a
 * host round trip. d_token_id may equal out_token.
 * Source: as mk_decode_step (megakernel and latency paragraphs of the
 * article); chaining the token on the device is this library's addition. */
int mk_decode_step_dev(mk_handle *h, const int32_t *d_token_id, int32_t position,
                       float *out_logits, int32_t *out_token, void *stream);

/* Same step through HOST buffers, for callers without device memory of their
 * own: the step reads *host_token and writes the greedy token to
 * *host_out_token (and the logits to host_logits if not NULL), then waits
 * for the stream. Pinned buffers the device can address (cudaHostAlloc'd or
 * registered) are read and written in place by the kernel over the chip
 * link; other host memory goes through copies on the stream (the logits
 * always do).
 * Source: as mk_decode_step; the host-buffer form is this library's
 * addition (the pages describe the device step only). */
int mk_decode_step_host(mk_handle *h, const int32_t *host_token, int32_t position,
                        float *host_logits, int32_t *host_out_token, void *stream);

/* One decode step for each of `batch` sequences (1 <= batch <= max_batch):
 * sequence b reads its token from d_tokens[b] and its position from
 * d_positions[b] (device int32 arrays, read when its step runs, so both can
 * be produced by the previous step on the device), attends over batch slot b
 * of the KV cache, appends its key/value row at its position, and writes its
 * greedy (or sampled, see mk_set_sampling) token to out_tokens[b] (device
 * int32[batch]) and, if out_logits is not NULL, its logits to
 * out_logits[b*vocab .. ] (device float[batch][vocab]).
 * With batch == max_batch and the fused batched step planned (see
 * mk_create), all sequences run through the last layer in ONE launch that
 * reads every layer's weight tile once for all of them; then three kernels
 * on the same stream form the final RMSNorm, the LM head (one tensor-core
 * contraction over the bf16 embedding for all sequences) and the draw. The
 * layer GEMVs take fp16 inputs, so the logits agree with the
 * single-sequence step to the parity tolerance, not bit for bit; a bounded
 * wait of the LM head that expired is reported by mk_get_status
 * (MK_ERR_TIMEOUT).
 * Otherwise the sequences run one fused step after another on `stream` (one
 * launch each, in batch order). A device token or position out of range is
 * reported by mk_get_status (MK_ERR_INVALID_ARG) and the step does nothing
 * for that sequence (the fused launch: for the whole batch).
 * Source: the article's internal-infrastructure paragraph (the same planned
 * sequences serve batch processing) and its megakernel paragraph on small
 * batch sizes and single sequences. */
int mk_decode_step_batch(mk_handle *h, const int32_t *d_tokens, const int32_t *d_positions, int32_t batch,
                         float *out_logits, int32_t *out_tokens, void *stream);

/* Multi-token prefill of batch slot 0: runs the n prompt tokens d_tokens[0 ..
 * n) (device int32[n]) at positions start_pos .. start_pos + n - 1 through
 * every layer at once, writes the key/value rows of all n positions into
 * the KV cache, and writes the logits of the last prompt position to
 * out_logits (device float[vocab], nullable) and the next token to out_token
 * (device int32[1]): greedy, or with sampling on (mk_set_sampling,
 * mk_set_sampling_filter) drawn as the decode step at that position would
 * draw it (the same noise and filter). The cache then holds what n consecutive
 * mk_decode_step calls would have left (to rounding), so decoding continues
 * at start_pos + n. The projections run as tensor-core contractions
 * (tcgen05.mma, bf16 weights x the activations split into two bf16 terms,
 * fp32 accumulation in tensor memory); attention is causal over the cache.
 * A few launches per layer on `stream` (asynchronous). The first call makes
 * the weights' tensor maps; a call with more tokens than any before
 * allocates the scratch for them (on the current device, owned by the
 * handle). MK_ERR_INVALID_ARG for a NULL pointer, n < 1 or positions past
 * max_seq; a prompt token outside [0, vocab) or an expired in-kernel wait is
 * reported by mk_get_status. One call in flight per handle, like the decode
 * steps (they share the cache).
 * Source: the article's internal-infrastructure paragraph (the planned
 * forward pass reused for batch processing): a prompt is such a batch, and
 * its projections are dense contractions. */
int mk_prefill(mk_handle *h, const int32_t *d_tokens, int32_t n, int32_t start_pos, float *out_logits,
               int32_t *out_token, void *stream);

/* The prefill's tensor-core contraction on its own:
 * d_y[n][m] = sum_k W[m][k] (Bhi[n][k] + Blo[n][k]) (+ d_r[n][m] if d_r is
 * not NULL; d_r may equal d_y) for m < M, n < N, with W = d_w bf16 [M][K],
 * Bhi = d_bhi and Blo = d_blo bf16 [N][K], d_y / d_r fp32 [N][M]; K a
 * multiple of 64, all pointers 16-byte aligned. d_status (device int32,
 * zeroed by the caller) becomes non-zero if an in-kernel wait expires.
 * Asynchronous on `stream`. Returns 0, -1 for bad arguments, -2 for a CUDA
 * error, -4 if the tensor maps cannot be made.
 * Source: as mk_prefill; a unit entry of this library for tests and
 * measurement. */
int mk_tc_gemm(const void *d_w, int32_t M, int32_t K, const void *d_bhi, const void *d_blo, int32_t N, float *d_y,
               const float *d_r, int32_t *d_status, void *stream);

/* The same step as a chain of separate kernel launches, one per stage
 * (QKV, attention, O-projection, gate/up, down per layer; LM head), with the
 * stream order between launches instead of in-kernel waits. Same results
 * bit for bit; exists to measure what fusing into one launch saves.
 * Source: the article's paragraphs on kernel launches and pipeline bubbles
 * (the many-small-kernels baseline the megakernel replaces); the glossary
 * entry "Megakernel" (synthszr.com), section on why the pauses between
 * compute steps are expensive. */
int mk_decode_step_unfused(mk_handle *h, int32_t token_id, int32_t position,
                           float *out_logits, int32_t *out_token, void *stream);

/* The decode step of mk_decode_step for callers that cannot allocate device
 * memory (a host framework that owns all device memory through its own pool,
 * a plugin that may only use the buffers it is handed, code that must not
 * trigger an allocation's implicit synchronisation). There is no handle: the
 * caller passes the model every call, and the kernel's scratch (instruction
 * queues, dependency counters, activations, attention partials, RoPE table)
 * lives in one file-scope device array of 16 MiB that every GPU loading this
 * library holds until the process exits. No counterpart in the megakernel
 * article: it is an interface addition of this library.
 *   - Allocates no device memory: no cudaMalloc, cudaFree or allocating
 *     library routine. Host-side planning uses ordinary host memory.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and plans and uploads
 *     the instruction queues; later calls with the same config, weight and
 *     cache pointers reuse them and only clear the counters before the
 *     launch. Make the first call (and any call with new inputs) before
 *     capturing a stream.
 *   - Every call shares the one array and it keeps the last call's contents;
 *     calls whose kernels overlap on the GPU (different streams, or a second
 *     model while the first still runs) race on it.
 *   - Returns MK_ERR_INVALID_ARG with a message if the model needs more
 *     scratch than the array holds (use mk_create then). A device-side wait
 *     timeout is not reported by this asynchronous call.
 * Arguments are those of mk_create plus those of mk_decode_step. */
int mk_decode_step_noalloc(const mk_config *config, const mk_weights *weights,
                           const mk_kv_cache *kv, int32_t token_id, int32_t position,
                           float *out_logits, int32_t *out_token, void *stream);

/* Device-side status of the last steps. Synchronises the handle's device,
 * returns MK_OK or MK_ERR_TIMEOUT (a bounded in-kernel wait expired; the step
 * that hit it produced undefined outputs) and resets it. After a timeout the
 * kernels refuse to run until this is called.
 * Source: the article's synchronisation paragraph (dependencies resolved by
 * counters in global memory inside the kernel); the pages say nothing about
 * failures, so a bounded wait and this status word are the library's own
 * failure mode for those in-kernel waits. */
int mk_get_status(mk_handle *h);

/* Bounded-wait limit for in-kernel dependency waits, in nanoseconds
 * (default 2e9). Host-only setting, takes effect on the next step.
 * Source: as mk_get_status (the synchronisation paragraph's in-kernel
 * waits); the limit itself is this library's convention. */
int mk_set_wait_timeout(mk_handle *h, uint64_t timeout_ns);

/* Sampling instead of greedy decoding for the following steps (all entry
 * points of this handle). temperature > 0: the returned token is a draw from
 * softmax(logits / temperature), taken as argmax_i(logit_i / temperature +
 * g_i) with Gumbel noise g_i = -log(-log(u_i)), u_i = (top 23 bits of word 0
 * of Philox4x32-10(counter {i, position, kv slot, 0}, key {seed low 32 bits,
 * seed high 32 bits}) + 1/2) / 2^23, which lies strictly inside (0, 1) for
 * every word — a counter-based draw, so a step is reproducible from (seed,
 * position, slot). temperature <= 0: greedy (the default). out_logits stay
 * the unscaled logits. Host-only setting; MK_ERR_INVALID_ARG for a
 * non-finite or vanishing temperature.
 * Source: the glossary entry "Megakernel" (synthszr.com), section on
 * megakernels in chatbots (token-by-token generation); the pages define no
 * sampler, so the draw follows two published definitions: the Gumbel-max
 * rule (Gumbel 1954) and Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11). */
int mk_set_sampling(mk_handle *h, float temperature, uint64_t seed);

/* Top-k / top-p filtering of the sampled draw for the following steps (all
 * entry points of this handle; it applies while mk_set_sampling's
 * temperature is > 0). The draw then chooses among a kept set only:
 *   1. candidates: the top_k largest logits (ties: the lower vocabulary
 *      index first); with top_k = 0 and top_p < 1, the MK_MAX_TOP_K largest;
 *   2. within them, e_j = exp((logit_j - max logit) / temperature); the kept
 *      set is the shortest prefix of the candidates whose sum of e_j reaches
 *      top_p times the candidates' total (at least one candidate);
 *   3. the token is argmax over the kept set of logit / temperature + g,
 *      with the Gumbel noise g of mk_set_sampling.
 * top_k = 0 and top_p = 1 (the default) switch filtering off. The sums run
 * in fp32. With a filter on, a fused batched step (mk_decode_step_batch)
 * draws every sequence's token with two short kernels after its LM head;
 * smaller batches run sequence by sequence as without a filter. A
 * single-sequence step draws in its LM-head epilogue, unless the model's LM
 * head has more than 256 blocks (the plan splits the vocabulary into more
 * instructions than the last block can sort the candidates of, e.g. a
 * 3B-class d_model of 3072): then the step writes its logits (to an
 * internal buffer if out_logits is NULL) and the same two kernels draw its
 * token, with the same noise. The candidate lists of that case are
 * allocated here (MK_ERR_NOMEM or MK_ERR_CUDA if that fails). MK_ERR_INVALID_ARG for top_k
 * outside [0, MK_MAX_TOP_K] or top_p outside (0, 1]. Host-only setting,
 * takes effect on the next step.
 * Source: the glossary entry "Megakernel" (synthszr.com), section on
 * megakernels in chatbots; the pages define no sampler, so the filter
 * follows the nucleus sampling of Holtzman, Buys, Du, Forbes, Choi (ICLR
 * 2020) with the customary top-k restriction before it. */
#define MK_MAX_TOP_K 64
int mk_set_sampling_filter(mk_handle *h, int32_t top_k, float top_p);

/* The sampling epilogue's random numbers on their own (no handle, no model):
 * for i = 0..n-1, word x_i = word 0 of Philox4x32-10(counter {i, position,
 * slot, 0}, key {seed low, seed high}) and noise g_i = -log(-log(u(x_i))),
 * with u as in mk_set_sampling, computed by the same device functions the
 * LM-head epilogue uses. If d_words (device uint32[n]) is not NULL, the
 * noise is computed from those words instead of Philox (to check chosen
 * words such as the all-ones word). Writes d_out_words (device uint32[n])
 * and d_out_noise (device float[n]) when not NULL; at least one must be
 * given. Asynchronous on `stream`; MK_ERR_INVALID_ARG for n < 0.
 * Source: as mk_set_sampling; a diagnostic of this library. */
int mk_sampling_noise(int32_t n, int32_t position, int32_t slot, uint64_t seed, const uint32_t *d_words,
                      uint32_t *d_out_words, float *d_out_noise, void *stream);

/* Tokens drawn from logits already on the device, by the kernels a fused
 * batched step (with a filter) and a sampled prefill run after their LM
 * head: for b = 0..batch-1, d_out_tokens[b] (device int32[batch]) is the
 * draw of mk_set_sampling at `temperature` from d_logits[b*vocab ..
 * (b+1)*vocab) (device float[batch][vocab]) with the noise of KV slot b at
 * position d_positions[b] (device int32[batch]), filtered as
 * mk_set_sampling_filter describes when top_k > 0 or top_p < 1. The library
 * keeps the kernels' scratch, grown as needed (not thread-safe).
 * Asynchronous on `stream`. MK_ERR_INVALID_ARG for NULL pointers, batch or
 * vocab < 1, temperature <= 0 or not finite, top_k outside [0,
 * MK_MAX_TOP_K] or top_p outside (0, 1].
 * Source: as mk_set_sampling_filter; a diagnostic of this library. */
int mk_draw_from_logits(const float *d_logits, int32_t batch, int32_t vocab, float temperature, int32_t top_k,
                        float top_p, const int32_t *d_positions, uint64_t seed, int32_t *d_out_tokens, void *stream);


/* ---- W2A8 GEMV: ternary weights, 8-bit activations ----------------------
 * The GEMV of the page "BitNet 1.58bit GPU Inference Kernel: Revolutionäre
 * Effizienz für KI-Modelle mit W2A8-Quantisierung" (dasgeld.co): 2-bit
 * weights and 8-bit activations, sixteen 2-bit values interleaved in each
 * 32-bit word, int8 dot products with dp4a. A weight matrix is
 * beta * Wq with Wq in {-1, 0, +1} [rows][cols] and one fp32 scale beta; the
 * input x is quantised per token, s = 127 / max(max|x|, 1e-5),
 * x_q = clamp(rint(x * s), -128, 127) in fp32, and
 * y[r] = beta / s * sum_c Wq[r][c] x_q[c] (exact integer sum, one fp32 scale).
 *
 * Packed layout (MK_W2 layout): row-major, cols / 16 uint32 words per row;
 * word w holds elements 16w .. 16w+15, element 16w + 4j + i (i, j in 0..3)
 * in bits [8i + 2j, 8i + 2j + 2) as the code Wq + 1 (code 3 is invalid). */

/* Host: packs q (int8 in {-1, 0, 1}, row-major [rows][cols], cols a multiple
 * of 16) into out (host uint32 [rows][cols / 16]). MK_ERR_INVALID_ARG for a
 * NULL pointer, cols % 16 != 0 or a value outside {-1, 0, 1}. */
int mk_w2_pack(const int8_t *q, int64_t rows, int64_t cols, uint32_t *out);

/* Host: the inverse of mk_w2_pack; MK_ERR_INVALID_ARG on an invalid code. */
int mk_w2_unpack(const uint32_t *packed, int64_t rows, int64_t cols, int8_t *q);

/* y = W2A8(packed, beta) x on the device: d_packed [rows][cols / 16] uint32
 * (16-byte aligned), d_x float[cols] (16-byte aligned), d_y float[rows];
 * cols one of 2048, 4096, 6144, 8192. One kernel launch on `stream`
 * (asynchronous); MK_ERR_INVALID_ARG for a bad pointer or size.
 * Source: the BitNet page above (its GEMV kernel, interleaved 2-bit packing,
 * dp4a); the quantisers follow BitNet b1.58 (Ma et al., 2024). */
int mk_w2a8_gemv(const uint32_t *d_packed, float beta, int32_t rows, int32_t cols, const float *d_x,
                 float *d_y, void *stream);

/* Activation-sparse down projection of one token: y = W_down h, where only
 * the hidden units with h_i != 0 are read. d_w_down_t: bf16 W_down
 * transposed, [F][d] (hidden unit i owns the contiguous row i, so a zero
 * unit costs no weight bytes); d_h: fp32 [F]; d_y: fp32 [d] (written). The
 * units are listed and their rows gathered per block of rows, and the
 * blocks' partial sums added in a fixed order: equal inputs give equal bits,
 * and the result is the dense product up to fp32 rounding order. d a
 * multiple of 8 up to 4096; weights and y 16-byte aligned.
 * Asynchronous on `stream`; the partial sums live in a workspace the unit
 * keeps (allocated on first use, grown for larger shapes). Returns 0, -1
 * (bad pointer, size or alignment), -3 (unsupported d), -4 (no workspace) or
 * -2 (launch failed).
 * Source: the TwELL article (iaexpertos.net, "Sakana AI und NVIDIA: TwELL
 * beschleunigt LLMs um bis zu 21,9 %"), sections on the sparsity GPUs ignore
 * and on kernels that process only the non-zero elements of an FFN layer;
 * the transposed ("twisted", one row per element) layout is the plain reading
 * of the name the article gives. */
int mk_twell_down(const void *d_w_down_t, int32_t F, int32_t d, const float *d_h, float *d_y, void *stream);

/* The ReLU-gated FFN of one token with the sparse down projection:
 * h = max(W_gate x, 0) * (W_up x) (W_gate, W_up bf16 [F][d], x fp32 [d],
 * h fp32 [F] written), then y = W_down h over the non-zero units as
 * mk_twell_down. d one of 256, 512, 1024, 2048, 3072, 4096; alignment and
 * return values as mk_twell_down.
 * Source: as mk_twell_down (a ReLU-type gate leaves most hidden units
 * exactly zero, the sparsity the article's kernels exploit). */
int mk_twell_ffn(const void *d_w_gate, const void *d_w_up, const void *d_w_down_t, int32_t F, int32_t d,
                 const float *d_x, float *d_h, float *d_y, void *stream);

/* Optional per-instruction timing: when `enable` is non-zero, every step
 * records %globaltimer stamps per instruction into a device buffer that
 * mk_read_trace copies out (see mk_read_trace).
 * Source: the article's closing paragraph (synchronisation overhead and
 * activation loading as the open costs): the trace measures exactly those
 * waits per instruction. */
int mk_set_trace(mk_handle *h, int32_t enable);

/* Copies the trace of the last traced step to host_out: records of 8 int64
 * {sm, instruction op, start - tile wait, start ns, phase0 ns, phase1 ns,
 * phase2 ns, end ns}, SM after SM in queue order; "tile wait" is the time
 * the instruction spent waiting for its weight / KV tiles to land. Phases of
 * a GEMV instruction: input polled (and normalised), tiles done, epilogue
 * written; of an attention instruction: q/k/v polled, tiles done, output
 * written. The last traced step is a single-sequence or a fused batched
 * step (mk_decode_step_batch), whichever ran last with tracing on. Returns
 * the number of records copied (or a negative status); cap = records that
 * fit in host_out. With host_out NULL, returns the number of records the
 * last traced step holds and copies nothing.
 * Source: as mk_set_trace. */
int mk_read_trace(mk_handle *h, int64_t *host_out, int32_t cap);

/* Diagnostics of a library built with MK_CHECKED (every device-side global
 * and shared-memory access is validated against the registered buffers; the
 * first violation is recorded and the access skipped). Copies the record
 * {site, address, bytes, (block << 32) | thread} to host_out4 (site 0 = none)
 * after synchronising the device. Returns 1 for a checked build, 0 for a
 * normal build (whose record is always zero), or a negative status.
 * Source: none on the pages; a diagnostic of this library. */
int mk_debug_read(mk_handle *h, uint64_t *host_out4);

/* Number of streaming multiprocessors (persistent CTAs) the plan uses and
 * the number of instructions in the plan.
 * Source: the article's internal-infrastructure paragraph (one instruction
 * sequence per SM). */
int mk_plan_size(const mk_handle *h, int32_t *n_sm, int32_t *n_instr);

/* Host-only, no device needed: plans the queues for `config` on `n_sm` SMs
 * and writes them out for inspection. With config->max_batch > 1 and a model
 * the fused batched step supports, this is the batched step's plan (ATTN
 * records then carry the sequence index in mat), else the single-sequence
 * plan. out_instr receives n_instr records of
 * MK_INSTR_WORDS int32 (queue order, SM after SM), out_queue_len[n_sm] the
 * queue lengths, *out_n_counters the number of dependency counters.
 * Returns the number of instructions, or a negative status if cap is too
 * small or the config is unsupported. Record layout:
 *   {op, layer, a0, a1, mat, wait_ctr, wait_target, sig_ctr, sig_n, stage,
 *    slot, bytes_lo, bytes_hi, 0, 0, 0}
 * op: 1 QKV, 2 ATTN, 3 OPROJ, 4 GATEUP, 5 DOWN, 6 LMHEAD. For GEMV ops
 * a0/a1 = first row / row count (QKV rows of the stacked [Wq; Wk; Wv],
 * mat = 0); for ATTN a0 = kv head, a1 = split index. The wait/signal fields
 * describe the dependency DAG as counts (wait_ctr < 0: no wait); the kernel
 * itself waits on the tagged activation words those producers write.
 * Source: the article's internal-infrastructure paragraph (sequences planned
 * on the host, one per SM) and synchronisation paragraph (counters that
 * tell an instruction when its inputs are ready). */
#define MK_INSTR_WORDS 16
int mk_plan_inspect(const mk_config *config, int32_t n_sm, int32_t *out_instr, int32_t cap,
                    int32_t *out_queue_len, int32_t *out_n_counters);

/* NULL-safe; waits for the device, then frees everything mk_create allocated.
 * Source: none; the pages are silent on resource lifetime, and this is the
 * boundary's own convention (the counterpart of mk_create). */
void mk_destroy(mk_handle *h);

/* Thread-local text of the last error ("" if none).
 * Source: none; the pages are silent on error reporting, and this is the
 * boundary's own convention. */
const char *mk_last_error(void);

#ifdef __cplusplus
}
#endif
#endif
