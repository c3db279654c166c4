// mk_kernel.cu — host-side launch helpers of the megakernel (called from
// mk_host.cpp): picks the instance for the model's head dimension and group
// size and launches it.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "mk_plan.h"

extern "C" const void *mk_kernel_fn_hd64(int G);
extern "C" const void *mk_kernel_fn_hd64_batch(int G);
extern "C" const void *mk_kernel_fn_hd128(int G);

namespace {
// instance for head dim hd (64 or 128), G query heads per kv head (1..4) and
// single-sequence or batched steps (batched: hd 64 only)
const void *kernel_for(int hd, int G, bool batch = false) {
    if (hd == 64) return batch ? mk_kernel_fn_hd64_batch(G) : mk_kernel_fn_hd64(G);
    if (hd == 128 && !batch) return mk_kernel_fn_hd128(G);
    return nullptr;
}
}  // namespace

extern "C" cudaError_t mk_kernel_configure(void) {
    for (int hd : {64, 128})
        for (int G = 1; G <= 4; ++G)
            for (bool batch : {false, true}) {
                const void *fn = kernel_for(hd, G, batch);
                if (!fn) continue;
                const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                           mk::kSmemBytes);
                if (e != cudaSuccess) return e;
            }
    return cudaSuccess;
}

extern "C" cudaError_t mk_kernel_launch(const mk::Params *p, int n_sm, int cooperative,
                                        cudaStream_t stream) {
    const void *fn = kernel_for(p->hd, p->attn_heads, p->nb > 1);
    if (!fn) return cudaErrorInvalidValue;
    void *args[] = {const_cast<mk::Params *>(p)};
    if (cooperative)
        return cudaLaunchCooperativeKernel(fn, dim3(n_sm), dim3(mk::kThreads), args, mk::kSmemBytes, stream);
    return cudaLaunchKernel(fn, dim3(n_sm), dim3(mk::kThreads), args, mk::kSmemBytes, stream);
}

extern "C" cudaError_t mk_kernel_occupancy(int *blocks_per_sm) {
    // every instance has the same block size and shared memory
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, kernel_for(64, 4), mk::kThreads,
                                                         mk::kSmemBytes);
}

namespace {
// bf16 -> fp16, round to nearest (exact for magnitudes in fp16's normal
// range); values whose magnitude exceeds fp16's largest finite value (which
// would become infinities) are counted in *out_of_range.
__global__ void bf16_to_f16(const uint16_t *__restrict__ src, uint16_t *__restrict__ dst, size_t n,
                            unsigned long long *out_of_range) {
    unsigned long long bad = 0;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const float v = __uint_as_float((uint32_t)src[i] << 16);
        const __half h = __float2half_rn(v);
        bad += (fabsf(v) <= 3.402823466e38f && __hisinf(h)) ? 1ull : 0ull;
        dst[i] = __half_as_ushort(h);
    }
    if (bad) atomicAdd(out_of_range, bad);
}
}  // namespace

// fp16 copy of n bf16 values (device pointers), on `stream`; out_of_range
// (device counter, nullable) accumulates the values beyond fp16's range.
extern "C" cudaError_t mk_convert_bf16_f16(const void *src, void *dst, size_t n, unsigned long long *out_of_range,
                                           cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    if (!out_of_range) return cudaErrorInvalidValue;
    bf16_to_f16<<<1024, 256, 0, stream>>>(static_cast<const uint16_t *>(src), static_cast<uint16_t *>(dst), n,
                                          out_of_range);
    return cudaGetLastError();
}
