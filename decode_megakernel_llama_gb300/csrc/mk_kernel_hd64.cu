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
