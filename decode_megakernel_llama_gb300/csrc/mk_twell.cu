// mk_twell.cu — activation-sparse FFN of one token, after the TwELL article
// (iaexpertos.net, "Sakana AI und NVIDIA: TwELL beschleunigt LLMs um bis zu
// 21,9 %"): kernels that process only the non-zero hidden units of an FFN
// block (unstructured activation sparsity, as a ReLU-type gate leaves it)
// instead of multiplying the zeros too.
//
// The down projection is read transposed, W_down^T [F][d]: hidden unit i owns
// the contiguous row i (d bf16 values), so a unit whose activation is zero
// costs no weight bytes at all and a non-zero one costs one 16-byte aligned
// row read with full bursts. Per call:
//   1. twell_part: CTA b takes R <= 32 rows and finds their non-zero units
//      with one ballot; each thread owns fixed columns of every row and
//      accumulates h_i * row_i over the non-zero rows, 8 or 16 rows' loads
//      in flight at a time, into part[b][.];
//   2. twell_reduce: y[c] = the sum of part[b][c] over b in a fixed order.
// The result is the dense product W_down h up to fp32 rounding order; equal
// inputs give equal bits.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr int kT = 256;            // threads per CTA
constexpr int kWarps = kT / 32;

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// 16 bytes of read-only weights, not kept in L1 (each is read once).
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Programmatic dependent launch (as in the prefill): the reduce may start
// while the row blocks finish, and a kernel waits for its predecessor's
// results with pdl_wait; without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Marks v as used here: called on every loaded vector after a batch of
// loads, it keeps the compiler from moving arithmetic between the loads, so
// a thread's loads are all in flight together.
__device__ __forceinline__ void pin(uint4 &v) { asm volatile("" : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)); }

// acc[e] += row chunk (8 bf16) * hv, as four packed pairs.
__device__ __forceinline__ void fma8(float2 (&acc)[4], const uint4 w, float hv) {
    const float2 h2 = make_float2(hv, hv);
    acc[0] = __ffma2_rn(make_float2(bf_lo(w.x), bf_hi(w.x)), h2, acc[0]);
    acc[1] = __ffma2_rn(make_float2(bf_lo(w.y), bf_hi(w.y)), h2, acc[1]);
    acc[2] = __ffma2_rn(make_float2(bf_lo(w.z), bf_hi(w.z)), h2, acc[2]);
    acc[3] = __ffma2_rn(make_float2(bf_lo(w.w), bf_hi(w.w)), h2, acc[3]);
}

// Partial sums of CTA b over rows [b*R, min(F, (b+1)*R)) of W_down^T, R <=
// 32. Thread t owns the 8-column chunks t and t + 256 (CPT of them) of every
// row, so a warp reads 512 contiguous bytes of a row per load and no two
// threads share an output: no shared memory, no barrier. Every warp loads the
// R activations (lane k the k-th), a ballot marks the non-zero ones, and the
// threads walk the set bits Q rows at a time with all of those rows' loads in
// flight together (16 rows, 64 KB per CTA, with one chunk a thread; 8 with two).
template <int CPT>
__global__ void __launch_bounds__(kT) twell_part(const uint16_t *__restrict__ wt, const float *__restrict__ h, int F,
                                                 int d, int R, float *__restrict__ part) {
    constexpr int Q = CPT == 1 ? 16 : 8;  // rows per batch of loads
    const int tid = threadIdx.x, lane = tid & 31;
    const int r0 = blockIdx.x * R, n = min(R, F - r0);
    const int nchunk = d / 8;
    pdl_wait();  // h may come from the kernel before (the FFN's gate/up)
    pdl_trigger();
    const float mine = lane < n ? h[r0 + lane] : 0.f;
    unsigned left = __ballot_sync(0xFFFFFFFFu, mine != 0.f);
    float2 acc[CPT][4];
#pragma unroll
    for (int c = 0; c < CPT; ++c)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[c][e] = make_float2(0.f, 0.f);
    while (left) {
        uint4 wv[Q][CPT];
        float hv[Q];
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            const int k = left ? __ffs(left) - 1 : -1;
            left = left ? left & (left - 1u) : 0u;
            const float v = __shfl_sync(0xFFFFFFFFu, mine, k < 0 ? 0 : k);
            hv[q] = k < 0 ? 0.f : v;
            const uint4 *row = reinterpret_cast<const uint4 *>(wt + (size_t)(r0 + (k < 0 ? 0 : k)) * d);
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                const int g = tid + c * kT;
                wv[q][c] = (k >= 0 && g < nchunk) ? ld_stream(row + g) : make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int q = 0; q < Q; ++q)
#pragma unroll
            for (int c = 0; c < CPT; ++c) pin(wv[q][c]);
#pragma unroll
        for (int q = 0; q < Q; ++q)
            if (hv[q] != 0.f)  // (warp-uniform) slots past the last non-zero row add nothing
#pragma unroll
                for (int c = 0; c < CPT; ++c) fma8(acc[c], wv[q][c], hv[q]);
    }
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        const int g = tid + c * kT;
        if (g < nchunk) {
            float4 *dst = reinterpret_cast<float4 *>(part + (size_t)blockIdx.x * d + (size_t)g * 8);
            dst[0] = make_float4(acc[c][0].x, acc[c][0].y, acc[c][1].x, acc[c][1].y);
            dst[1] = make_float4(acc[c][2].x, acc[c][2].y, acc[c][3].x, acc[c][3].y);
        }
    }
}

// y[c] = sum over b < nb of part[b][c]: a CTA of 32 warps takes 32 columns;
// warp s sums the blocks b = s, s + 32, ... of its lane's column, and the 32
// slice sums of a column are added in slice order.
constexpr int kRT = 1024;
__global__ void __launch_bounds__(kRT) twell_reduce(const float *__restrict__ part, int nb, int D, float *__restrict__ y) {
    __shared__ float ss[kRT / 32][33];
    pdl_wait();  // the row blocks' partial sums
    pdl_trigger();
    const int lane = threadIdx.x & 31, s = threadIdx.x >> 5;
    const int c = blockIdx.x * 32 + lane;
    float acc = 0.f;
    if (c < D) {
        // the slice's blocks 16 at a time, all 16 loads in flight before any add
        for (int b0 = s; b0 < nb; b0 += 16 * (kRT / 32)) {
            float v[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int b = b0 + u * (kRT / 32);
                v[u] = b < nb ? part[(size_t)b * D + c] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 16; ++u) acc += v[u];
        }
    }
    ss[s][lane] = acc;
    __syncthreads();
    if (threadIdx.x < 32 && c < D) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kRT / 32; ++w) t += ss[w][lane];
        y[c] = t;
    }
}

// Hidden activations of a ReLU-gated FFN: h_i = max(g_i, 0) * u_i with
// g = W_gate x, u = W_up x (bf16 [F][d], x fp32 [d]); one warp per unit,
// both rows' loads in flight together, lane l owning chunks k*32 + l.
template <int NC>
__global__ void __launch_bounds__(kT) twell_gateup(const uint16_t *__restrict__ wg, const uint16_t *__restrict__ wu,
                                                   const float *__restrict__ x, int F, float *__restrict__ h) {
    constexpr int D = NC * 256;
    __shared__ float4 xs[D / 4];
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int i = tid; i < D / 4; i += kT) xs[i] = reinterpret_cast<const float4 *>(x)[i];
    __syncthreads();
    const int i = blockIdx.x * kWarps + warp;
    if (i >= F) return;
    const uint4 *ga = reinterpret_cast<const uint4 *>(wg + (size_t)i * D) + lane;
    const uint4 *ua = reinterpret_cast<const uint4 *>(wu + (size_t)i * D) + lane;
    uint4 gw[NC], uw[NC];
#pragma unroll
    for (int k = 0; k < NC; ++k) {
        gw[k] = ld_stream(ga + k * 32);
        uw[k] = ld_stream(ua + k * 32);
    }
#pragma unroll
    for (int k = 0; k < NC; ++k) {
        pin(gw[k]);
        pin(uw[k]);
    }
    float2 g2 = make_float2(0.f, 0.f), u2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < NC; ++k) {
        const float4 x0 = xs[(k * 32 + lane) * 2], x1 = xs[(k * 32 + lane) * 2 + 1];
        const float2 xp[4] = {make_float2(x0.x, x0.y), make_float2(x0.z, x0.w), make_float2(x1.x, x1.y),
                              make_float2(x1.z, x1.w)};
        const uint32_t gu[4] = {gw[k].x, gw[k].y, gw[k].z, gw[k].w};
        const uint32_t uu[4] = {uw[k].x, uw[k].y, uw[k].z, uw[k].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            g2 = __ffma2_rn(make_float2(bf_lo(gu[e]), bf_hi(gu[e])), xp[e], g2);
            u2 = __ffma2_rn(make_float2(bf_lo(uu[e]), bf_hi(uu[e])), xp[e], u2);
        }
    }
    float g = g2.x + g2.y, u = u2.x + u2.y;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        g += __shfl_xor_sync(0xFFFFFFFFu, g, o);
        u += __shfl_xor_sync(0xFFFFFFFFu, u, o);
    }
    if (lane == 0) h[i] = g > 0.f ? g * u : 0.f;
}

template <int CPT>
cudaError_t launch_part(const uint16_t *wt, const float *h, int F, int d, int R, int nb, float *part, cudaStream_t s) {
    return launch_pdl(twell_part<CPT>, dim3(nb), dim3(kT), 0, s, wt, h, F, d, R, part);
}

template <int NC>
cudaError_t launch_gateup(const uint16_t *wg, const uint16_t *wu, const float *x, int F, float *h, cudaStream_t s) {
    return launch_pdl(twell_gateup<NC>, dim3((F + kWarps - 1) / kWarps), dim3(kT), 0, s, wg, wu, x, F, h);
}

// Rows per CTA of the down projection: about two CTAs per SM, at most 32
// (one activation per lane).
int rows_per_cta(int F, int n_sm) {
    int R = (F + 2 * n_sm - 1) / (2 * n_sm);
    return R < 1 ? 1 : (R > 32 ? 32 : R);
}

// Widths of the FFN entry (its gate/up kernel is instantiated per width).
int check_d(int d) {
    switch (d) {
        case 256: case 512: case 1024: case 2048: case 3072: case 4096: return 0;
        default: return -3;
    }
}

// Widths of the down projection: 16-byte rows, at most two chunks a thread.
int check_d_down(int d) { return (d >= 8 && d % 8 == 0 && d / 8 <= 2 * kT) ? 0 : -3; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The K-split partials live in a workspace this unit keeps (grown when a
// larger shape needs more; freed at exit).
float *workspace(size_t floats) {
    static float *work = nullptr;
    static size_t have = 0;
    if (floats > have) {
        if (work) {
            cudaDeviceSynchronize();
            cudaFree(work);
        }
        work = nullptr;
        have = 0;
        if (cudaMalloc(&work, floats * sizeof(float)) == cudaSuccess) have = floats;
    }
    return work;
}

cudaError_t down(const uint16_t *wt, int F, int d, const float *h, float *y, cudaStream_t s, int *rc) {
    int dev = 0, n_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorInvalidDevice;
    const int R = rows_per_cta(F, n_sm), nb = (F + R - 1) / R;
    float *part = workspace((size_t)nb * d);
    if (!part) {
        *rc = -4;
        return cudaErrorMemoryAllocation;
    }
    const cudaError_t e = d / 8 <= kT ? launch_part<1>(wt, h, F, d, R, nb, part, s)
                                      : launch_part<2>(wt, h, F, d, R, nb, part, s);
    if (e != cudaSuccess) return e;
    return launch_pdl(twell_reduce, dim3((d + 31) / 32), dim3(kRT), 0, s, part, nb, d, y);
}

}  // namespace

// y = W_down h over the non-zero entries of h only (see the file comment).
extern "C" int mk_twell_down(const void *d_w_down_t, int32_t F, int32_t d, const float *d_h, float *d_y,
                             void *stream) {
    if (!d_w_down_t || !d_h || !d_y || F < 1) return -1;
    if (check_d_down(d)) return -3;
    if (!aligned16(d_w_down_t) || !aligned16(d_y)) return -1;
    int rc = -2;
    const cudaError_t e = down(static_cast<const uint16_t *>(d_w_down_t), F, d, d_h, d_y,
                               static_cast<cudaStream_t>(stream), &rc);
    return e == cudaSuccess ? 0 : rc;
}

// The ReLU-gated FFN of one token: h = max(W_gate x, 0) * (W_up x), then
// y = W_down h over the non-zero units of h.
extern "C" int mk_twell_ffn(const void *d_w_gate, const void *d_w_up, const void *d_w_down_t, int32_t F, int32_t d,
                            const float *d_x, float *d_h, float *d_y, void *stream) {
    if (!d_w_gate || !d_w_up || !d_w_down_t || !d_x || !d_h || !d_y || F < 1) return -1;
    if (check_d(d)) return -3;
    if (!aligned16(d_w_gate) || !aligned16(d_w_up) || !aligned16(d_w_down_t) || !aligned16(d_x) || !aligned16(d_y))
        return -1;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint16_t *wg = static_cast<const uint16_t *>(d_w_gate), *wu = static_cast<const uint16_t *>(d_w_up);
    cudaError_t e;
    switch (d / 256) {
        case 1: e = launch_gateup<1>(wg, wu, d_x, F, d_h, s); break;
        case 2: e = launch_gateup<2>(wg, wu, d_x, F, d_h, s); break;
        case 4: e = launch_gateup<4>(wg, wu, d_x, F, d_h, s); break;
        case 8: e = launch_gateup<8>(wg, wu, d_x, F, d_h, s); break;
        case 12: e = launch_gateup<12>(wg, wu, d_x, F, d_h, s); break;
        default: e = launch_gateup<16>(wg, wu, d_x, F, d_h, s); break;
    }
    if (e != cudaSuccess) return -2;
    int rc = -2;
    e = down(static_cast<const uint16_t *>(d_w_down_t), F, d, d_h, d_y, s, &rc);
    return e == cudaSuccess ? 0 : rc;
}
