// mk_kernel_hd64.cu — megakernel instances for head dimension 64
// (G = 1..4 query heads per kv head), compiled as their own translation unit.
#include "mk_kernel.cuh"

extern "C" const void *mk_kernel_fn_hd64(int G) {
    switch (G) {
        case 1: return (const void *)mk::mk_megakernel<64, 1, false>;
        case 2: return (const void *)mk::mk_megakernel<64, 2, false>;
        case 3: return (const void *)mk::mk_megakernel<64, 3, false>;
        case 4: return (const void *)mk::mk_megakernel<64, 4, false>;
        default: return nullptr;
    }
}

// Batched-step instances (hd 64 only).
extern "C" const void *mk_kernel_fn_hd64_batch(int G) {
    switch (G) {
        case 1: return (const void *)mk::mk_megakernel<64, 1, true>;
        case 2: return (const void *)mk::mk_megakernel<64, 2, true>;
        case 3: return (const void *)mk::mk_megakernel<64, 3, true>;
        case 4: return (const void *)mk::mk_megakernel<64, 4, true>;
        default: return nullptr;
    }
}

// ---------------------------------------------------------------------------
// The sampling epilogue's noise on its own: word 0 of Philox4x32-10 and the
// Gumbel noise for vocabulary entries 0..n-1, through the same device
// functions the LM-head epilogue calls (so a test can compare the kernel's
// stream with an independent implementation, and feed chosen words).
// ---------------------------------------------------------------------------
namespace {
__global__ void mk_noise_kernel(int n, int pos, int slot, uint32_t seed_lo, uint32_t seed_hi,
                                const uint32_t *words, uint32_t *out_words, float *out_noise) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const uint32_t x = words ? words[i]
                                 : mk::philox_w0((uint32_t)i, (uint32_t)pos, (uint32_t)slot, 0u, seed_lo, seed_hi);
        if (out_words) out_words[i] = x;
        if (out_noise) out_noise[i] = mk::gumbel_from_word(x);
    }
}
}  // namespace

extern "C" cudaError_t mk_noise_launch(int n, int pos, int slot, uint64_t seed, const uint32_t *words,
                                       uint32_t *out_words, float *out_noise, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const int blocks = (n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024;
    mk_noise_kernel<<<blocks, 256, 0, stream>>>(n, pos, slot, (uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32),
                                                words, out_words, out_noise);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Draws from logits [B][V] already in memory, for a fused batched step with a
// top-k / top-p filter (its LM head writes every sequence's logits) and for a
// prefill's last position: sequence b draws with KV slot b's noise at
// position positions[b] (positions NULL: pos0). Filtered:
//   filter_lists: CTA (slice j, sequence b) keys entries [1024 j, 1024 j +
//     1024) of sequence b's logits and publishes its top_k best, in order, as
//     list j of sequence b;
//   filter_draw: CTA b draws sequence b's token from its lists with the
//     single-sequence epilogue's own tail (draw_filtered).
// Plain (temperature only): sample_slices keys logit / T + noise per slice
// and keeps the slice's best; sample_reduce takes the best of the slices.
// ---------------------------------------------------------------------------
namespace {
constexpr int kFilterSlice = 1024;

__global__ void __launch_bounds__(mk::kConsumerThreads) filter_lists(const float *logits, int V, int K,
                                                                     unsigned long long *lists) {
    __shared__ unsigned long long keys[kFilterSlice];
    const int b = blockIdx.y, j = blockIdx.x, base = j * kFilterSlice;
    const float *lg = logits + (size_t)b * V;
    for (int i = threadIdx.x; i < kFilterSlice; i += blockDim.x) {
        const int e = base + i;
        keys[i] = e < V ? mk::argmax_key(lg[e], (uint32_t)e) : 0ull;  // no real key is 0
    }
    mk::consumer_sync();
    mk::block_top64(keys, kFilterSlice);
    unsigned long long *mine = lists + ((size_t)b * gridDim.x + j) * mk::kMaxTopK;
    for (int t = threadIdx.x; t < K; t += blockDim.x) mine[t] = keys[t];
}

__global__ void __launch_bounds__(mk::kConsumerThreads) filter_draw(const unsigned long long *lists, int nl, int K,
                                                                    float top_p, float inv_temp,
                                                                    const int32_t *positions, int pos0, int slot0,
                                                                    uint32_t seed_lo, uint32_t seed_hi,
                                                                    int32_t *out_tokens) {
    extern __shared__ unsigned long long g[];  // max(nl * K, 64) keys
    __shared__ int gcount;
    const int b = blockIdx.x;
    const int pos = positions ? positions[b] : pos0;
    const int tok = mk::draw_filtered(lists + (size_t)b * nl * mk::kMaxTopK, nl, K, top_p, inv_temp, pos,
                                      slot0 + b, seed_lo, seed_hi, g, &gcount);
    if (threadIdx.x == 0) out_tokens[b] = tok;
}

// inv_temp > 0: the key of logit * inv_temp + noise; otherwise of the logit
// itself (the greedy choice, lowest index on ties).
__global__ void __launch_bounds__(256) sample_slices(const float *logits, int V, float inv_temp,
                                                     const int32_t *positions, int pos0, uint32_t seed_lo,
                                                     uint32_t seed_hi, unsigned long long *keys) {
    __shared__ unsigned long long best8[8];
    const int b = blockIdx.y, j = blockIdx.x, base = j * kFilterSlice;
    const int pos = positions ? positions[b] : pos0;
    const float *lg = logits + (size_t)b * V;
    unsigned long long best = 0ull;
    for (int i = threadIdx.x; i < kFilterSlice; i += blockDim.x) {
        const int e = base + i;
        if (e < V) {
            const float z = inv_temp > 0.f ? lg[e] * inv_temp + mk::gumbel_noise((uint32_t)e, pos, b, seed_lo, seed_hi)
                                           : lg[e];
            const unsigned long long k = mk::argmax_key(z, (uint32_t)e);
            best = k > best ? k : best;
        }
    }
    best = mk::warp_max_u64(best);
    if ((threadIdx.x & 31) == 0) best8[threadIdx.x >> 5] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 0; w < 8; ++w) best = best8[w] > best ? best8[w] : best;
        keys[(size_t)b * gridDim.x + j] = best;
    }
}

// The final RMSNorm of a batched step's residual stream (x of sequence b at
// bofs(b, e), fp32) with gains g, as the hi / lo bf16 terms [b][d] of the
// LM head's input: a CTA per sequence.
__global__ void __launch_bounds__(256) batch_final_norm(const float *x, int d, const uint16_t *g, float eps,
                                                        uint16_t *hi, uint16_t *lo) {
    __shared__ float red[8];
    const int b = blockIdx.x;
    float ss = 0.f;
    for (int e = threadIdx.x; e < d; e += blockDim.x) {
        const float v = x[mk::bofs(b, e)];
        ss = fmaf(v, v, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    ss = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) ss += red[w];
    const float r = 1.0f / sqrtf(ss / (float)d + eps);
    for (int e = threadIdx.x; e < d; e += blockDim.x) {
        const float v = x[mk::bofs(b, e)] * (r * mk::bf16f(g[e]));
        const uint16_t h = mk::f2bf(v);
        hi[(size_t)b * d + e] = h;
        lo[(size_t)b * d + e] = mk::f2bf(v - mk::bf16f(h));
    }
}

__global__ void __launch_bounds__(32) sample_reduce(const unsigned long long *keys, int ns, int32_t *out_tokens) {
    const int b = blockIdx.x;
    unsigned long long best = 0ull;
    for (int j = threadIdx.x; j < ns; j += 32) best = keys[(size_t)b * ns + j] > best ? keys[(size_t)b * ns + j] : best;
    best = mk::warp_max_u64(best);
    if (threadIdx.x == 0) out_tokens[b] = (int32_t)mk::key_index(best);
}
}  // namespace

// Lists of the filtered draw of a batch: B * ceil(V / 1024) * kMaxTopK keys.
extern "C" size_t mk_filter_lists_keys(int B, int V) {
    return (size_t)B * ((V + kFilterSlice - 1) / kFilterSlice) * mk::kMaxTopK;
}

extern "C" cudaError_t mk_filtered_draw_batch(const float *logits, int B, int V, int K, float top_p, float inv_temp,
                                              const int32_t *positions, int pos0, int slot0, uint64_t seed,
                                              unsigned long long *lists, int32_t *out_tokens, cudaStream_t stream) {
    if (B < 1 || V < 1 || K < 1 || K > mk::kMaxTopK) return cudaErrorInvalidValue;
    const int nl = (V + kFilterSlice - 1) / kFilterSlice;
    const size_t smem = (size_t)(nl * K > 64 ? nl * K : 64) * sizeof(unsigned long long);
    static size_t configured = 0;
    if (smem > configured) {
        const cudaError_t e = cudaFuncSetAttribute(filter_draw, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = smem;
    }
    filter_lists<<<dim3(nl, B), mk::kConsumerThreads, 0, stream>>>(logits, V, K, lists);
    filter_draw<<<B, mk::kConsumerThreads, smem, stream>>>(lists, nl, K, top_p, inv_temp, positions, pos0, slot0,
                                                           (uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32),
                                                           out_tokens);
    return cudaGetLastError();
}

// The plain draw (temperature, no filter; inv_temp = 0: the greedy choice)
// of B sequences from their logits; keys: B * ceil(V / 1024) slots of scratch.
extern "C" cudaError_t mk_sampled_draw_batch(const float *logits, int B, int V, float inv_temp,
                                             const int32_t *positions, int pos0, uint64_t seed,
                                             unsigned long long *keys, int32_t *out_tokens, cudaStream_t stream) {
    if (B < 1 || V < 1 || !(inv_temp >= 0.f)) return cudaErrorInvalidValue;
    const int ns = (V + kFilterSlice - 1) / kFilterSlice;
    sample_slices<<<dim3(ns, B), 256, 0, stream>>>(logits, V, inv_temp, positions, pos0, (uint32_t)(seed & 0xFFFFFFFFu),
                                                   (uint32_t)(seed >> 32), keys);
    sample_reduce<<<B, 32, 0, stream>>>(keys, ns, out_tokens);
    return cudaGetLastError();
}

// The final RMSNorm of a batched step's B sequences into the LM head's hi /
// lo bf16 input [B][d].
extern "C" cudaError_t mk_batch_final_norm(const float *x, int B, int d, const uint16_t *gain, float eps, uint16_t *hi,
                                           uint16_t *lo, cudaStream_t stream) {
    if (B < 1 || B > mk::kMaxBatch || d < 1) return cudaErrorInvalidValue;
    batch_final_norm<<<B, 256, 0, stream>>>(x, d, gain, eps, hi, lo);
    return cudaGetLastError();
}
