// mk_w2a8.cu — the W2A8 GEMV: ternary weights packed sixteen to a 32-bit
// word, 8-bit activations, integer dot products with dp4a.
//
// "BitNet 1.58bit GPU Inference Kernel: Revolutionäre Effizienz für
// KI-Modelle mit W2A8-Quantisierung" (dasgeld.co) describes a GEMV kernel
// with 2-bit weights and 8-bit activations: sixteen 2-bit values interleaved
// in one 32-bit integer so that they decode in parallel, and the dp4a
// instruction for the 4-element int8 dot products. The page gives no
// formulas; the quantisers are BitNet b1.58's: a weight matrix is beta * Wq
// with Wq in {-1, 0, +1} and one fp32 scale beta, and the input x is
// quantised per token by its absolute maximum,
//     s = 127 / max(max|x|, 1e-5),  x_q = clamp(rint(x * s), -128, 127),
// so y[r] = beta / s * sum_c Wq[r][c] x_q[c].
//
// Packed layout (this library's; the page's own block permutation is not
// printed): row r is cols / 16 words; word w holds elements 16w .. 16w+15,
// element 16w + 4j + i in bits [8i + 2j, 8i + 2j + 2) as the code Wq + 1.
// (word >> 2j) & 0x03030303 then holds the codes of elements 16w + 4j ..
// 16w + 4j + 3 in its four bytes, the operand layout of dp4a against four
// consecutive int8 activations; sum_c (code - 1) x_q = dp4a sums - sum x_q.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mk.h"

namespace {

constexpr int kW2Warps = 8;
constexpr int kW2Threads = kW2Warps * 32;
constexpr int kW2Rows = 8;  // rows of a batch (one 16-byte chunk of each per lane); two batches in flight

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Streams the weights once: no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// dp4a with unsigned bytes in a and signed bytes in b.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// One 16-byte chunk (4 words, 64 elements) against its 16 words of codes.
// The codes of bit pair j are taken in place, word & (0x03030303 << 2j):
// bytes code * 4^j (at most 128, hence unsigned bytes), so pair j's products
// sum to 4^j times its dot product. The four sums are exact integers and
// shift back without remainder: no shift per word.
__device__ __forceinline__ int dot_chunk(const uint4 w, const uint32_t (&xq)[16], int acc) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    int a[4] = {0, 0, 0, 0};
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int j = 0; j < 4; ++j) a[j] = dp4a_us(ws[m] & (0x03030303u << (2 * j)), xq[4 * m + j], a[j]);
    return acc + a[0] + (a[1] >> 2) + (a[2] >> 4) + (a[3] >> 6);
}

// Reduce-scatter of 8 per-lane integers over the warp: afterwards lane l
// holds the warp sum of value (l >> 2) & 7 (9 shuffles for 8 rows).
__device__ __forceinline__ int warp_reduce8(const int (&a)[8]) {
    const int lane = threadIdx.x & 31;
    const bool h16 = (lane & 16) != 0, h8 = (lane & 8) != 0, h4 = (lane & 4) != 0;
    int b[4], c[2];
#pragma unroll
    for (int v = 0; v < 4; ++v) b[v] = (h16 ? a[v + 4] : a[v]) + __shfl_xor_sync(0xFFFFFFFFu, h16 ? a[v] : a[v + 4], 16);
#pragma unroll
    for (int v = 0; v < 2; ++v) c[v] = (h8 ? b[v + 2] : b[v]) + __shfl_xor_sync(0xFFFFFFFFu, h8 ? b[v] : b[v + 2], 8);
    int e = (h4 ? c[1] : c[0]) + __shfl_xor_sync(0xFFFFFFFFu, h4 ? c[0] : c[1], 4);
    e += __shfl_xor_sync(0xFFFFFFFFu, e, 2);
    return e + __shfl_xor_sync(0xFFFFFFFFu, e, 1);
}

// cols = KS * 2048. A row is KS slices of 2048 elements; warp (rg, ks) of a
// block takes slice ks of kW2Rows rows at a time (row group rg), so each
// lane holds the 64 activation codes of one 16-byte weight chunk in 16
// registers and has kW2Rows chunks in flight. The slices' integer sums meet
// in shared memory (exact), and one scale turns them into y.
template <int KS>
__global__ void __launch_bounds__(kW2Threads, 2) w2a8_gemv_kernel(const uint4 *__restrict__ W, float beta, int rows,
                                                                 const float *__restrict__ x, float *__restrict__ y) {
    constexpr int K = KS * 2048;
    constexpr int RG = kW2Warps / KS;  // row groups per block (warps beyond RG * KS idle)
    __shared__ float wmax[kW2Warps];
    __shared__ int part[kW2Warps][kW2Rows];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rg = warp / KS, ks = warp % KS;
    const bool active = rg < RG;
    // per-token absmax of x (every block computes it: x is K floats)
    float am = 0.f;
    for (int i = tid; i < K; i += kW2Threads) am = fmaxf(am, fabsf(x[i]));
    am = warp_max_f(am);
    if (lane == 0) wmax[warp] = am;
    __syncthreads();
    am = 0.f;
#pragma unroll
    for (int w = 0; w < kW2Warps; ++w) am = fmaxf(am, wmax[w]);
    const float s = 127.0f / fmaxf(am, 1e-5f);
    // this lane's activation codes: elements ks * 2048 + lane * 64 .. +64
    uint32_t xq[16];
    int xs = 0;
    {
        const float4 *src = reinterpret_cast<const float4 *>(x + ks * 2048 + lane * 64);
#pragma unroll
        for (int w = 0; w < 16; ++w) {
            const float4 v = src[w];
            const float f[4] = {v.x, v.y, v.z, v.w};
            uint32_t word = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int q = (int)fminf(fmaxf(rintf(f[i] * s), -128.f), 127.f);
                xs += q;
                word |= (uint32_t)(q & 0xFF) << (8 * i);
            }
            xq[w] = word;
        }
    }
    xs = warp_sum_i(xs);  // the slice's code sum
    const float fscale = beta / s;
    // rows in batches of kW2Rows per warp; the next batch's loads go out
    // before the current batch is multiplied (two batches in flight)
    const int step = gridDim.x * RG * kW2Rows;
    auto load_batch = [&](int r0, uint4 (&wv)[kW2Rows]) {
        const int rb = r0 + rg * kW2Rows;
#pragma unroll
        for (int k = 0; k < kW2Rows; ++k) {
            const int r = rb + k < rows ? rb + k : rows - 1;
            wv[k] = ld_stream(W + (size_t)r * (K / 64) + ks * 32 + lane);
        }
    };
    uint4 cur[kW2Rows], nxt[kW2Rows];
    int r0 = blockIdx.x * RG * kW2Rows;
    if (active && r0 < rows) load_batch(r0, cur);
    for (; r0 < rows; r0 += step) {
        if (active) {
            if (r0 + step < rows) load_batch(r0 + step, nxt);
            int acc[kW2Rows];
#pragma unroll
            for (int k = 0; k < kW2Rows; ++k) acc[k] = dot_chunk(cur[k], xq, 0);
            const int sum = warp_reduce8(acc);
            if ((lane & 3) == 0) part[warp][lane >> 2] = sum - xs;
#pragma unroll
            for (int k = 0; k < kW2Rows; ++k) cur[k] = nxt[k];
        }
        __syncthreads();
        if (tid < RG * kW2Rows) {
            const int g = tid / kW2Rows, k = tid % kW2Rows, r = r0 + g * kW2Rows + k;
            int tot = 0;
#pragma unroll
            for (int q = 0; q < KS; ++q) tot += part[g * KS + q][k];
            if (r < rows) y[r] = (float)tot * fscale;
        }
        __syncthreads();
    }
}

template <int KS>
cudaError_t launch_ks(const uint4 *W, float beta, int rows, const float *x, float *y, int grid, cudaStream_t s) {
    w2a8_gemv_kernel<KS><<<grid, kW2Threads, 0, s>>>(W, beta, rows, x, y);
    return cudaGetLastError();
}

}  // namespace

extern "C" {

int mk_w2_pack(const int8_t *q, int64_t rows, int64_t cols, uint32_t *out) {
    if (!q || !out || rows < 0 || cols < 0 || cols % 16) return MK_ERR_INVALID_ARG;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t w = 0; w < cols / 16; ++w) {
            uint32_t word = 0;
            for (int e = 0; e < 16; ++e) {
                const int v = q[r * cols + 16 * w + e];
                if (v < -1 || v > 1) return MK_ERR_INVALID_ARG;
                const int j = e / 4, i = e % 4;
                word |= (uint32_t)(v + 1) << (8 * i + 2 * j);
            }
            out[r * (cols / 16) + w] = word;
        }
    return MK_OK;
}

int mk_w2_unpack(const uint32_t *packed, int64_t rows, int64_t cols, int8_t *q) {
    if (!packed || !q || rows < 0 || cols < 0 || cols % 16) return MK_ERR_INVALID_ARG;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t w = 0; w < cols / 16; ++w) {
            const uint32_t word = packed[r * (cols / 16) + w];
            for (int e = 0; e < 16; ++e) {
                const int j = e / 4, i = e % 4;
                const int code = (int)((word >> (8 * i + 2 * j)) & 3u);
                if (code == 3) return MK_ERR_INVALID_ARG;
                q[r * cols + 16 * w + e] = (int8_t)(code - 1);
            }
        }
    return MK_OK;
}

int mk_w2a8_gemv(const uint32_t *d_packed, float beta, int32_t rows, int32_t cols, const float *d_x, float *d_y,
                 void *stream) {
    if (!d_packed || !d_x || !d_y || rows < 1 || cols < 2048 || cols % 2048 || cols > 8192)
        return MK_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(d_packed) | reinterpret_cast<uintptr_t>(d_x)) & 15u) return MK_ERR_INVALID_ARG;
    int dev = 0, n_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return MK_ERR_CUDA;
    const int ks = cols / 2048;
    const int per_block = (kW2Warps / ks) * kW2Rows;
    int grid = (rows + per_block - 1) / per_block;
    if (grid > 2 * n_sm) grid = 2 * n_sm;  // two resident blocks per SM, rows strided over them
    const uint4 *W = reinterpret_cast<const uint4 *>(d_packed);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (ks) {
        case 1: e = launch_ks<1>(W, beta, rows, d_x, d_y, grid, s); break;
        case 2: e = launch_ks<2>(W, beta, rows, d_x, d_y, grid, s); break;
        case 3: e = launch_ks<3>(W, beta, rows, d_x, d_y, grid, s); break;
        default: e = launch_ks<4>(W, beta, rows, d_x, d_y, grid, s); break;
    }
    return e == cudaSuccess ? MK_OK : MK_ERR_CUDA;
}

}  // extern "C"
