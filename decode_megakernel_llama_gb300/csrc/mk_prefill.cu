// mk_prefill.cu — multi-token prefill: the prompt's projections as tensor-core
// contractions (tcgen05), causal attention over the prompt, and the KV-cache
// rows of every prompt position, in a handful of launches per layer.
//
// The megakernel article ("Revolution der KI-Beschleunigung: Wie ein
// Low-Latency Megakernel den Llama-1B Turbo zündet", dasgeld.co, paragraph on
// the internal infrastructure) plans the forward pass once and reuses it for
// batch processing; a prompt of n tokens is such a batch. Its projections are
// real dense contractions Y[n][out] = X[n][in] W[out][in]^T, so they run on
// the 5th-generation tensor cores:
//   * the weights are the MMA's A operand (M = 128 output features per CTA),
//     the prompt's activations the B operand (N = 32 .. 128 tokens per CTA);
//   * both arrive by TMA (cp.async.bulk.tensor) as 128-byte-swizzled K-major
//     tiles of 64 elements into a ring of 4 to 8 shared-memory stages with
//     full/empty mbarriers;
//   * one thread issues tcgen05.mma (kind::f16, bf16 x bf16 -> fp32) into an
//     accumulator in tensor memory; tcgen05.commit frees a stage when its
//     MMAs are done;
//   * the epilogue reads the accumulator with tcgen05.ld and writes fp32
//     (adding the residual where the layer has one).
// The activations enter as two bf16 terms, hi = bf16(x) and lo = bf16(x -
// hi): x is then carried to about 16 significant bits, so the prefill meets
// the decode step's parity bar while the weights stay in their stored bf16.
// A stage holds the hi tile and the lo tile back to back, so one MMA with
// N = 2 BN multiplies the weight tile by both (hi in accumulator columns
// 0 .. BN-1, lo in BN .. 2BN-1, added in the epilogue): the loop is bound by
// the count of MMA instructions (a near-fixed cost each at these sizes), and
// this halves it.
//
// The causal attention over the prompt (attend_prefill_mma) also runs on the
// tensor cores, with warp-level mma.sync (its softmax sits between two small
// products per 64-position tile, row by row in registers): queries and
// probabilities enter as hi / lo bf16 terms, keys and values are the cache's
// bf16 rows.
//
// Every wait is bounded (%globaltimer, 2 s); on expiry the kernel records an
// error in a status word, still drains its copies and frees its tensor
// memory, and returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "mk_prefill.h"

namespace mkpf {
namespace {

constexpr int kThreads = 128;  // 4 warps: TMA issuer, MMA issuer, and all four for the epilogue
constexpr int kRingBytes = 196608;  // the stage ring: 192 KB of shared memory
constexpr int kATileBytes = 128 * 128;  // 128 rows x 64 bf16
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kMaxSplits = 16;

__device__ __forceinline__ uint32_t saddr(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

// Programmatic dependent launch: the prefill's kernels are launched so that
// the next one in the stream may start once every CTA of the current one has
// called pdl_trigger (or exited); it does its set-up (and a contraction its
// first weight-tile loads, which depend on nothing earlier) and then
// pdl_wait()s, which returns once the previous grid has completed and its
// writes are visible. Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(saddr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on an mbarrier phase; false (and the error word set) on expiry
// or when another thread of the grid already gave up.
__device__ bool mbar_wait(uint64_t *bar, uint32_t parity, int *err) {
    uint64_t t0 = 0;
    for (uint32_t it = 1;; ++it) {
        if (mbar_try(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*(volatile int *)err) return false;
            const uint64_t now = gtimer();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > kWaitNs) {
                atomicExch(err, 1);
                return false;
            }
        }
    }
}

// TMA: one box of a 2-D tensor map into shared memory, completing bytes on bar.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            saddr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(saddr(bar))
        : "memory");
}

// Shared-memory matrix descriptor of a K-major bf16 tile in the 128-byte
// swizzle layout that TMA writes: rows of 128 bytes (64 elements), atoms of 8
// rows every 1024 bytes along M (or N). Fields: start address >> 4 (bits
// 0-13), leading byte offset >> 4 (16-29; unused by this layout), stride
// byte offset >> 4 (32-45), the fixed 0b001 (46-48), base offset 0 (the
// tiles are 1024-byte aligned), swizzle mode 2 = 128 bytes (61-63). The k-th
// 16-element slice of a row starts 32 bytes further.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_byte_addr) {
    uint64_t d = (uint64_t)((smem_byte_addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1),
// A and B bf16 (7-9 = 1, 10-12 = 1), both K-major (15, 16 = 0), N >> 3
// (17-22), M >> 4 (24-28); M = 128, N <= 256.
template <int N>
__device__ __forceinline__ constexpr uint32_t idesc_bf16_f32() {
    static_assert(N % 16 == 0 && N >= 16 && N <= 256, "M = 128 needs N a multiple of 16 up to 256");
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives on bar once every MMA this thread issued before has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Y[n][m] (+)= sum_k W[m][k] (Bhi[n][k] + Blo[n][k]) for m < M, n < N:
// W [M][K] bf16 (tensor map ta, box 64 x 128), Bhi / Blo [N][K] bf16 (tensor
// maps tbh / tbl, box 64 x BN), Y and R fp32 with row stride ldy (R may be
// Y: an in-place residual add; or NULL). CTA (i, j) computes rows
// 128i .. 128i+127 of W for tokens BN*j .. BN*j+BN-1. K % 64 == 0.
// ---------------------------------------------------------------------------
// Stages of the ring for a token tile of BN: as many as fit in kRingBytes
// (8 for BN 32, 6 for 64, 4 for 128), so that enough TMA copies are in
// flight to hide their latency behind the MMAs.
template <int BN>
__host__ __device__ constexpr int stages_for() {
    return kRingBytes / (kATileBytes + 2 * BN * 128) > 8 ? 8 : kRingBytes / (kATileBytes + 2 * BN * 128);
}

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// fp32 -> bf16, round to nearest even (finite values).
__device__ __forceinline__ uint16_t f2bf_rne(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7F800000u) == 0x7F800000u) return uint16_t((u >> 16) | ((u & 0xFFFFu) ? 0x40u : 0u));
    u += 0x7FFFu + ((u >> 16) & 1u);
    return uint16_t(u >> 16);
}

// Up to three weight matrices multiplied by the same activations in one
// launch: CTA row tiles 0 .. tiles[0]-1 take matrix 0 (tensor map ta0),
// the next tiles[1] matrix 1 (ta1), then matrix 2 (ta2); each has its own
// rows, output and residual. With a K split the partial sums of split z go
// to part[z][N][mtot], matrix q's rows from column off[q].
struct Segs {
    int n;
    int tiles[3], M[3], ldy[3];
    float *Y[3];
    const float *R[3];
    int mtot, off[3];
    uint16_t *hhi, *hlo;  // gated launches: the hi / lo bf16 terms of h [N][ldy[0]]
};

// GATED: the gate/up projection of the MLP. A CTA takes 64 outputs: its A
// tile is 64 rows of W_gate (ta0, boxes of 64 rows) over 64 rows of W_up
// (ta1) for the same outputs, so the accumulator holds g in lanes 0..63 and u
// in lanes 64..127; the epilogue passes u through shared memory and writes
// h = silu(g) * u as the hi / lo bf16 terms the down projection reads.
template <int BN, bool GATED = false>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm(const __grid_constant__ CUtensorMap ta0, const __grid_constant__ CUtensorMap ta1,
            const __grid_constant__ CUtensorMap ta2, const __grid_constant__ CUtensorMap tbh,
            const __grid_constant__ CUtensorMap tbl, const Segs sg, int N, int K, float *part, int *err) {
    constexpr int kBTileBytes = BN * 128;
    constexpr int kStageBytes = kATileBytes + 2 * kBTileBytes;
    constexpr int kStages = stages_for<BN>();
    constexpr uint32_t kCols = 2 * BN < 32 ? 32 : 2 * BN;  // tensor-memory columns: hi, then lo (a power of two >= 32)
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + kStages * kStageBytes);
    uint64_t *empty = full + kStages;
    uint64_t *done = empty + kStages;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(done + 1);
    int *issued = reinterpret_cast<int *>(tslot + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int bx = blockIdx.x, q = 0;
    if (!GATED)
        while (q + 1 < sg.n && bx >= sg.tiles[q]) bx -= sg.tiles[q++];
    const CUtensorMap *ta = q == 0 ? &ta0 : (q == 1 ? &ta1 : &ta2);
    const int M = sg.M[q];
    float *Y = sg.Y[q];
    int ldy = sg.ldy[q];
    const float *R = sg.R[q];
    const int m0 = bx * (GATED ? 64 : 128), n0 = blockIdx.y * BN;
    // K split over gridDim.z CTAs: this one takes 64-wide chunks c0 .. c0+nk-1
    // and writes its partial sums to part[z][N][mtot] (summed later in a
    // fixed order), or with one split the result itself
    const int nk_all = K / 64, z = blockIdx.z, S = gridDim.z;
    const int c0 = z * nk_all / S, nk = (z + 1) * nk_all / S - c0;
    if (S > 1) {
        Y = part + (size_t)z * N * sg.mtot + sg.off[q];
        ldy = sg.mtot;
        R = nullptr;
    }
    // the A tile of chunk kc into stage memory st (gated: gate rows, then up rows)
    auto load_a = [&](uint8_t *st, int kc, uint64_t *bar) {
        if (GATED) {
            tma_load_2d(st, &ta0, (c0 + kc) * 64, m0, bar);
            tma_load_2d(st + kATileBytes / 2, &ta1, (c0 + kc) * 64, m0, bar);
        } else {
            tma_load_2d(st, ta, (c0 + kc) * 64, m0, bar);
        }
    };
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        *issued = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tslot)),
                     "r"(kCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    // the weight tiles of the first stages do not depend on the previous
    // kernel: their copies go out before the wait for its results
    const int pre = nk < kStages ? nk : kStages;
    if (warp == 0 && lane == 0)
        for (int kc = 0; kc < pre; ++kc) {
            mbar_expect_tx(&full[kc], kStageBytes);
            load_a(sm + kc * kStageBytes, kc, &full[kc]);
        }
    pdl_wait();
    pdl_trigger();

    if (warp == 0 && lane == 0) {
        // TMA issuer: the activations of the first stages, then stage s of
        // chunk kc once the MMAs of chunk kc - kStages freed it
        for (int kc = 0; kc < pre; ++kc) {
            uint8_t *st = sm + kc * kStageBytes;
            tma_load_2d(st + kATileBytes, &tbh, (c0 + kc) * 64, n0, &full[kc]);
            tma_load_2d(st + kATileBytes + kBTileBytes, &tbl, (c0 + kc) * 64, n0, &full[kc]);
            *issued = kc + 1;
        }
        for (int kc = pre; kc < nk; ++kc) {
            const int s = kc % kStages;
            if (!mbar_wait(&empty[s], ((kc / kStages) - 1) & 1, err)) break;
            uint8_t *st = sm + s * kStageBytes;
            mbar_expect_tx(&full[s], kStageBytes);
            load_a(st, kc, &full[s]);
            tma_load_2d(st + kATileBytes, &tbh, (c0 + kc) * 64, n0, &full[s]);
            tma_load_2d(st + kATileBytes + kBTileBytes, &tbl, (c0 + kc) * 64, n0, &full[s]);
            *issued = kc + 1;
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer: 4 k-slices of 16 per chunk; B = the hi tile and the lo
        // tile that follows it (2 BN rows), one MMA for both terms
        constexpr uint32_t idesc = idesc_bf16_f32<2 * BN>();
        bool ok = true;
        for (int kc = 0; kc < nk && ok; ++kc) {
            const int s = kc % kStages;
            ok = mbar_wait(&full[s], (kc / kStages) & 1, err);
            if (!ok) break;
            tc_fence_after();
            const uint32_t a = saddr(sm + s * kStageBytes), bh = a + kATileBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                umma_bf16(tmem, sw128_desc(a + kk * 32), sw128_desc(bh + kk * 32), idesc, (kc | kk) != 0);
            umma_commit(&empty[s]);
        }
        if (ok) umma_commit(done);
    }
    __syncwarp();
    // epilogue: warp w reads tensor-memory lanes 32w .. 32w+31 (output rows)
    const bool have = mbar_wait(done, 0, err);
    tc_fence_after();
    if (GATED) {
        // g sits in tensor-memory lanes 0..63 (warps 0, 1), u in lanes 64..127
        // (warps 2, 3), row r of each in lane r and r + 64. Each warp hands the
        // half of its columns the partner warp finishes to shared memory, then
        // forms h for the other half: gate warps columns 0 .. BN/2-1, up
        // warps the rest. Every copy has landed and every MMA is done, so the
        // stage ring is free.
        constexpr int kH = BN / 2, kUs = kH + 1;  // padded rows: the lanes of a warp hit 32 banks
        static_assert(2 * 64 * kUs * 4 <= kStages * kStageBytes, "g and u do not fit the stage ring");
        float *us = reinterpret_cast<float *>(sm);  // [64][kUs] u of columns 0 .. kH-1
        float *gs = us + 64 * kUs;                  // [64][kUs] g of columns kH .. BN-1
        const bool up = warp >= 2;
        const int r = (warp & 1) * 32 + lane;
        const uint32_t row = tmem + ((uint32_t)(warp * 32) << 16);
        if (have) {
            const uint32_t cb = up ? 0 : kH;
            float *dst = (up ? us : gs) + r * kUs;
#pragma unroll 1
            for (int c = 0; c < kH; c += 16) {
                uint32_t vh[16], vl[16];
                tmem_ld16(row + cb + (uint32_t)c, vh);
                tmem_ld16(row + (uint32_t)BN + cb + (uint32_t)c, vl);
#pragma unroll
                for (int i = 0; i < 16; ++i) dst[c + i] = __uint_as_float(vh[i]) + __uint_as_float(vl[i]);
            }
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (have) {
            const int cb = up ? kH : 0, m = m0 + r;
            const float *oth = (up ? gs : us) + r * kUs;
#pragma unroll 1
            for (int c = 0; c < kH; c += 16) {
                uint32_t vh[16], vl[16];
                tmem_ld16(row + (uint32_t)(cb + c), vh);
                tmem_ld16(row + (uint32_t)(BN + cb + c), vl);
                if (m < M) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int n = n0 + cb + c + i;
                        if (n < N) {
                            const float mine = __uint_as_float(vh[i]) + __uint_as_float(vl[i]), o = oth[c + i];
                            const float g = up ? o : mine, u = up ? mine : o;
                            const float v = g / (1.0f + expf(-g)) * u;
                            const uint16_t hb = f2bf_rne(v);
                            sg.hhi[(size_t)n * ldy + m] = hb;
                            sg.hlo[(size_t)n * ldy + m] = f2bf_rne(v - bf2f(hb));
                        }
                    }
                }
            }
        }
    } else if (have) {
        const int m = m0 + warp * 32 + lane;
        const uint32_t row = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
        for (int c = 0; c < BN; c += 16) {
            uint32_t vh[16], vl[16];
            tmem_ld16(row + (uint32_t)c, vh);
            tmem_ld16(row + (uint32_t)(BN + c), vl);
            if (m < M) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int n = n0 + c + i;
                    if (n < N) {
                        float y = __uint_as_float(vh[i]) + __uint_as_float(vl[i]);
                        if (R) y += R[(size_t)n * ldy + m];
                        Y[(size_t)n * ldy + m] = y;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        // a failed CTA still lets its issued copies land before its shared memory goes
        const int ni = *issued, lo = ni > kStages ? ni - kStages : 0;
        for (int kc = lo; kc < ni; ++kc) {
            const uint64_t t0 = gtimer();
            while (!mbar_try(&full[kc % kStages], (kc / kStages) & 1))
                if (gtimer() - t0 > kWaitNs) break;
        }
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols) : "memory");
    }
}

// Y[n][m] = R[n][m] (if any) + sum over z of part[z][n][m], z in order.
__global__ void sum_splits(const float *part, int S, int N, int M, float *Y, int ldy, const float *R) {
    pdl_wait();
    pdl_trigger();
    const size_t total = (size_t)N * M;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const size_t n = i / M, m = i % M;
        float y = R ? R[n * ldy + m] : 0.f;
        for (int z = 0; z < S; ++z) y += part[(size_t)z * total + i];
        Y[n * ldy + m] = y;
    }
}

// Launches a prefill kernel with programmatic stream serialization (see
// pdl_wait): it may start while the previous kernel of the stream finishes.
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

template <int BN>
constexpr int gemm_smem_bytes() {
    return stages_for<BN>() * (kATileBytes + 2 * BN * 128) + 1024 + 256;
}

// ---------------------------------------------------------------------------
// Elementwise and attention kernels of the prefill.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float block_sum(float v, float *red) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    float t = 0.f;
    for (int i = 0; i < nw; ++i) t += red[i];
    return t;
}

// X[t] = float(E[tokens[t]]); a token outside [0, V) sets the error word.
__global__ void embed_rows(const uint16_t *E, const int32_t *tokens, int n, int d, int V, float *X, int *err) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    const int tok = tokens[t];
    if (tok < 0 || tok >= V) {
        if (threadIdx.x == 0) atomicExch(err, 2);
        return;
    }
    for (int i = threadIdx.x; i < d; i += blockDim.x) X[(size_t)t * d + i] = bf2f(E[(size_t)tok * d + i]);
}

// hi/lo bf16 terms of rows of X [rows][K] (fp32), optionally RMSNorm'd with gain g.
__global__ void norm_split(const float *X, int K, const uint16_t *g, float eps, uint16_t *hi, uint16_t *lo) {
    __shared__ float red[32];
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    const float *x = X + (size_t)t * K;
    float scale = 1.f;
    if (g) {
        float ss = 0.f;
        for (int i = threadIdx.x; i < K; i += blockDim.x) ss = fmaf(x[i], x[i], ss);
        ss = block_sum(ss, red);
        scale = 1.0f / sqrtf(ss / (float)K + eps);
    }
    for (int i = threadIdx.x; i < K; i += blockDim.x) {
        const float v = g ? x[i] * (scale * bf2f(g[i])) : x[i];
        const uint16_t h = f2bf_rne(v);
        hi[(size_t)t * K + i] = h;
        lo[(size_t)t * K + i] = f2bf_rne(v - bf2f(h));
    }
}

// The split sum of a residual contraction followed by the next RMSNorm:
// for token n = blockIdx.x, Y[n][m] = R[n][m] + sum over z of part[z][n][m]
// (z in order), then the RMSNorm of that row with gains g (as norm_split)
// into hi / lo bf16 terms [n][M]. A thread keeps kSnE elements (M <=
// kSnE * kSnThreads) and loads eight splits' partials of them before it adds
// any, so a pass waits for about one memory round trip per eight splits.
constexpr int kSnThreads = 512, kSnE = 8;

__global__ void __launch_bounds__(kSnThreads) sum_splits_norm(const float *__restrict__ part, int S, int N, int M,
                                                              float *__restrict__ Y, int ldy,
                                                              const float *__restrict__ R,
                                                              const uint16_t *__restrict__ g, float eps,
                                                              uint16_t *__restrict__ hi, uint16_t *__restrict__ lo) {
    __shared__ float red[32];
    pdl_wait();
    pdl_trigger();
    const int n = blockIdx.x, tid = threadIdx.x;
    const size_t total = (size_t)N * M;
    const float *pn = part + (size_t)n * M;
    float v[kSnE];
#pragma unroll
    for (int e = 0; e < kSnE; ++e) {
        const int m = tid + e * kSnThreads;
        v[e] = R && m < M ? R[(size_t)n * ldy + m] : 0.f;
    }
    for (int z0 = 0; z0 < S; z0 += 8) {
        float w[8][kSnE];
#pragma unroll
        for (int dz = 0; dz < 8; ++dz)
#pragma unroll
            for (int e = 0; e < kSnE; ++e) {
                const int m = tid + e * kSnThreads;
                w[dz][e] = z0 + dz < S && m < M ? pn[(size_t)(z0 + dz) * total + m] : 0.f;
            }
#pragma unroll
        for (int dz = 0; dz < 8; ++dz)
#pragma unroll
            for (int e = 0; e < kSnE; ++e)
                if (z0 + dz < S) v[e] += w[dz][e];
    }
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < kSnE; ++e) {
        const int m = tid + e * kSnThreads;
        if (m < M) {
            Y[(size_t)n * ldy + m] = v[e];
            ss = fmaf(v[e], v[e], ss);
        }
    }
    ss = block_sum(ss, red);
    const float scale = 1.0f / sqrtf(ss / (float)M + eps);
#pragma unroll
    for (int e = 0; e < kSnE; ++e) {
        const int m = tid + e * kSnThreads;
        if (m < M) {
            const float x = v[e] * (scale * bf2f(g[m]));
            const uint16_t h = f2bf_rne(x);
            hi[(size_t)n * M + m] = h;
            lo[(size_t)n * M + m] = f2bf_rne(x - bf2f(h));
        }
    }
}

// RoPE on q and k of token t (position pos0 + t) from the fp32 QKV rows, q
// kept (rotated) in place, bf16 k and v written into the cache at the position.
// With S > 0 the q|k|v row is first summed from the K-split partials
// part[z][t][.] (z in order): q's sums go to QKV (rotated), k's and v's to
// the cache as above. The blocks of a token (gridDim.y of them) share its
// pairs.
__global__ void rope_append(float *__restrict__ QKV, const float *__restrict__ part, int S, int n, int Hq, int Hkv,
                            int hd, int pos0, const float *__restrict__ rope, int max_seq, uint16_t *__restrict__ kc,
                            uint16_t *__restrict__ vc) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x, pos = pos0 + t;
    const int stride = (Hq + 2 * Hkv) * hd, half = hd / 2;
    float *row = QKV + (size_t)t * stride;
    const size_t zs = (size_t)n * stride;
    const float *prow = part + (size_t)t * stride;
    auto get = [&](int col) {
        if (S == 0) return row[col];
        float v = 0.f;
        for (int z = 0; z < S; ++z) v += prow[z * zs + col];
        return v;
    };
    const int first = blockIdx.y * blockDim.x + threadIdx.x, step = gridDim.y * blockDim.x;
    for (int idx = first; idx < (Hq + Hkv) * half; idx += step) {
        const int h = idx / half, i = idx % half;
        const int ca = h * hd + i, cb = ca + half;
        const float c = rope[((size_t)pos * half + i) * 2], s = rope[((size_t)pos * half + i) * 2 + 1];
        const float a = get(ca), b = get(cb);
        const float ra = a * c - b * s, rb = b * c + a * s;
        if (h < Hq) {
            row[ca] = ra;
            row[cb] = rb;
        } else {
            const int kvh = h - Hq;
            const size_t off = ((size_t)kvh * max_seq + pos) * hd;
            kc[off + i] = f2bf_rne(ra);
            kc[off + i + half] = f2bf_rne(rb);
        }
    }
    for (int idx = first; idx < Hkv * hd; idx += step) {
        const int kvh = idx / hd, i = idx % hd;
        vc[((size_t)kvh * max_seq + pos) * hd + i] = f2bf_rne(get((Hq + Hkv) * hd + idx));
    }
}

// Causal attention of the prompt on the tensor cores (mma.sync m16n8k16,
// bf16 operands, fp32 accumulators), flash-attention style. CTA (kv head,
// block of QB = 64 / G prompt tokens) holds 64 query rows, row r = (token
// t0 + r / G, query head kvh * G + r % G); warp w owns rows 16w .. 16w+15.
// Keys and values go through shared memory in tiles of 64 positions (rows
// padded by 16 bytes: conflict-free fragment loads). Per tile a warp forms
// S = (q/sqrt(hd)) K^T from the hi and lo bf16 terms of its scaled queries
// (two MMAs per fragment), masks the positions past each row's own, updates
// the rows' running max and sum (online softmax) and adds P V with P as hi
// and lo bf16 terms; V's fragments come from ldmatrix.trans. The output goes
// out as the hi / lo bf16 terms the O-projection reads.
constexpr int kFaWarps = 4;
constexpr int kFaRows = kFaWarps * 16;
constexpr int kFaKeys = 64;

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// bf16 pair (lo element first) of the high terms of (x, y); their low terms in *lo.
__device__ __forceinline__ uint32_t split2(float x, float y, uint32_t *lo) {
    const uint16_t hx = f2bf_rne(x), hy = f2bf_rne(y);
    *lo = (uint32_t)f2bf_rne(x - bf2f(hx)) | ((uint32_t)f2bf_rne(y - bf2f(hy)) << 16);
    return (uint32_t)hx | ((uint32_t)hy << 16);
}

template <int HD>
__global__ void __launch_bounds__(kFaWarps * 32) attend_prefill_mma(const float *__restrict__ QKV, int n, int Hq,
                                                                    int Hkv, int pos0, int max_seq,
                                                                    const uint16_t *__restrict__ kc,
                                                                    const uint16_t *__restrict__ vc,
                                                                    uint16_t *__restrict__ out_hi,
                                                                    uint16_t *__restrict__ out_lo) {
    constexpr int RS = HD + 8;       // padded row of a staged tile, in bf16
    constexpr int KSTEPS = HD / 16;  // k-steps of S = Q K^T
    constexpr int NT = HD / 8;       // n-tiles of O
    __shared__ __align__(16) uint16_t Ks[kFaKeys * RS], Vs[kFaKeys * RS];
    pdl_wait();
    pdl_trigger();
    const int kvh = blockIdx.x, G = Hq / Hkv, QB = kFaRows / G;
    const int t0 = blockIdx.y * QB;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
    const int stride = (Hq + 2 * Hkv) * HD;
    // this lane's two rows (g and g + 8 of the warp's 16)
    int T[2], tok[2], head[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int r = warp * 16 + g + 8 * hr;
        tok[hr] = t0 + r / G;
        head[hr] = kvh * G + r % G;
        const bool live = r < QB * G && tok[hr] < n;
        T[hr] = live ? pos0 + tok[hr] + 1 : 0;
    }
    // the scaled queries as A fragments, hi and lo terms
    uint32_t qh[KSTEPS][4], ql[KSTEPS][4];
    {
        const float scale = rsqrtf((float)HD);
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const float *q = T[hr] ? QKV + (size_t)tok[hr] * stride + (size_t)head[hr] * HD : nullptr;
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks)
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int col = ks * 16 + 2 * c + 8 * half;
                    const float x = q ? q[col] * scale : 0.f, y = q ? q[col + 1] * scale : 0.f;
                    qh[ks][hr + 2 * half] = split2(x, y, &ql[ks][hr + 2 * half]);
                }
        }
    }
    float o[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m[2] = {-1e30f, -1e30f}, l[2] = {0.f, 0.f};
    const int Tblk = pos0 + min(n, t0 + QB);  // positions the block's rows see
    const int Twarp = max(T[0], T[1]);        // (per lane; the warp's max below)
    int Tw = Twarp;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) Tw = max(Tw, __shfl_xor_sync(0xFFFFFFFFu, Tw, off));
    const uint4 *Kg = reinterpret_cast<const uint4 *>(kc + (size_t)kvh * max_seq * HD);
    const uint4 *Vg = reinterpret_cast<const uint4 *>(vc + (size_t)kvh * max_seq * HD);
    constexpr int CPR = HD / 8;
    for (int k0 = 0; k0 < Tblk; k0 += kFaKeys) {
        const int kn = min(kFaKeys, Tblk - k0);
        __syncthreads();
        for (int i = tid; i < kFaKeys * CPR; i += blockDim.x) {
            const int r = i / CPR, cc = i % CPR;
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4 *>(Ks + r * RS + cc * 8) = r < kn ? Kg[(size_t)(k0 + r) * CPR + cc] : z;
            *reinterpret_cast<uint4 *>(Vs + r * RS + cc * 8) = r < kn ? Vg[(size_t)(k0 + r) * CPR + cc] : z;
        }
        __syncthreads();
        if (k0 >= Tw) continue;  // past every row of this warp
        // S = Q K^T for the 64 positions (8 n-tiles of 8)
        float sc[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
            const uint16_t *kr = Ks + (j * 8 + g) * RS + 2 * c;
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) {
                const uint32_t b0 = *reinterpret_cast<const uint32_t *>(kr + ks * 16);
                const uint32_t b1 = *reinterpret_cast<const uint32_t *>(kr + ks * 16 + 8);
                mma_bf16(sc[j], qh[ks], b0, b1);
                mma_bf16(sc[j], ql[ks], b0, b1);
            }
        }
        // mask, running max and sum, P
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int hr = e >> 1, key = k0 + j * 8 + 2 * c + (e & 1);
                if (key >= T[hr]) sc[j][e] = -INFINITY;
                mx[hr] = fmaxf(mx[hr], sc[j][e]);
            }
        float corr[2];
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xFFFFFFFFu, mx[hr], 1));
            mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xFFFFFFFFu, mx[hr], 2));
            const float mn = fmaxf(m[hr], mx[hr]);
            corr[hr] = __expf(m[hr] - mn);
            m[hr] = mn;
        }
        float ps[2] = {0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int hr = e >> 1;
                sc[j][e] = __expf(sc[j][e] - m[hr]);  // masked: exp(-inf) = 0
                ps[hr] += sc[j][e];
            }
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            ps[hr] += __shfl_xor_sync(0xFFFFFFFFu, ps[hr], 1);
            ps[hr] += __shfl_xor_sync(0xFFFFFFFFu, ps[hr], 2);
            l[hr] = l[hr] * corr[hr] + ps[hr];
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            o[j][0] *= corr[0];
            o[j][1] *= corr[0];
            o[j][2] *= corr[1];
            o[j][3] *= corr[1];
        }
        // O += P V: k-step s covers positions 16s .. 16s+15 (n-tiles 2s, 2s+1 of S)
#pragma unroll
        for (int s2 = 0; s2 < 4; ++s2) {
            uint32_t ph[4], pl[4];
            ph[0] = split2(sc[2 * s2][0], sc[2 * s2][1], &pl[0]);
            ph[1] = split2(sc[2 * s2][2], sc[2 * s2][3], &pl[1]);
            ph[2] = split2(sc[2 * s2 + 1][0], sc[2 * s2 + 1][1], &pl[2]);
            ph[3] = split2(sc[2 * s2 + 1][2], sc[2 * s2 + 1][3], &pl[3]);
            // lane l addresses row (l % 8) + 8 ((l / 8) & 1) of the tile, columns 8 (l / 16) on
            const uint16_t *vrow = Vs + (s2 * 16 + (lane & 7) + 8 * ((lane >> 3) & 1)) * RS + 8 * (lane >> 4);
#pragma unroll
            for (int j = 0; j < NT; j += 2) {
                uint32_t b[4];
                asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                             : "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3])
                             : "r"(saddr(vrow + j * 8)));
                mma_bf16(o[j], ph, b[0], b[1]);
                mma_bf16(o[j], pl, b[0], b[1]);
                mma_bf16(o[j + 1], ph, b[2], b[3]);
                mma_bf16(o[j + 1], pl, b[2], b[3]);
            }
        }
    }
    // O / l as hi / lo bf16 terms
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        if (!T[hr]) continue;
        const float inv = 1.0f / l[hr];
        const size_t at = ((size_t)tok[hr] * Hq + head[hr]) * HD + 2 * c;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            uint32_t lo;
            const uint32_t hi = split2(o[j][2 * hr] * inv, o[j][2 * hr + 1] * inv, &lo);
            *reinterpret_cast<uint32_t *>(out_hi + at + j * 8) = hi;
            *reinterpret_cast<uint32_t *>(out_lo + at + j * 8) = lo;
        }
    }
}

// Final RMSNorm of one row into shared memory, then rows of the tied
// embedding times it (a warp per row), logits and a block argmax key.
__global__ void lm_head_rows(const float *x, const uint16_t *g, float eps, const uint16_t *E, int V, int d,
                             float *logits, unsigned long long *keys) {
    extern __shared__ float xs[];
    __shared__ float red[32];
    __shared__ unsigned long long best[32];
    pdl_wait();
    pdl_trigger();
    float ss = 0.f;
    for (int i = threadIdx.x; i < d; i += blockDim.x) ss = fmaf(x[i], x[i], ss);
    ss = block_sum(ss, red);
    const float r = 1.0f / sqrtf(ss / (float)d + eps);
    for (int i = threadIdx.x; i < d; i += blockDim.x) xs[i] = x[i] * (r * bf2f(g[i]));
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    unsigned long long bk = 0ull;
    for (int row = blockIdx.x * nw + warp; row < V; row += gridDim.x * nw) {
        const uint16_t *w = E + (size_t)row * d;
        float acc = 0.f;
        for (int c = lane * 8; c < d; c += 256) {
            const uint4 v = *reinterpret_cast<const uint4 *>(w + c);
            const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc = fmaf(__uint_as_float(u[e] << 16), xs[c + 2 * e], acc);
                acc = fmaf(__uint_as_float(u[e] & 0xFFFF0000u), xs[c + 2 * e + 1], acc);
            }
        }
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
        if (lane == 0) {
            if (logits) logits[row] = acc;
            uint32_t u = __float_as_uint(acc);
            u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
            const unsigned long long k = ((unsigned long long)u << 32) | (0xFFFFFFFFu - (uint32_t)row);
            bk = k > bk ? k : bk;
        }
    }
    if (lane == 0) best[warp] = bk;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long b = 0ull;
        for (int i = 0; i < nw; ++i) b = best[i] > b ? best[i] : b;
        keys[blockIdx.x] = b;
    }
}

__global__ void argmax_keys(const unsigned long long *keys, int n, int32_t *out_token) {
    __shared__ unsigned long long best[32];
    pdl_wait();
    pdl_trigger();
    unsigned long long b = 0ull;
    for (int i = threadIdx.x; i < n; i += blockDim.x) b = keys[i] > b ? keys[i] : b;
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long x = __shfl_xor_sync(0xFFFFFFFFu, b, o);
        b = x > b ? x : b;
    }
    if ((threadIdx.x & 31) == 0) best[threadIdx.x >> 5] = b;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) b = best[i] > b ? best[i] : b;
        *out_token = (int32_t)(0xFFFFFFFFu - (uint32_t)(b & 0xFFFFFFFFull));
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// Tensor map of a row-major bf16 matrix [rows][K], boxes of 64 x box_rows,
// 128-byte swizzle (rows past the end read as zeros).
bool encode_map(CUtensorMap *map, const void *ptr, int rows, int K, int box_rows) {
    EncodeTiledFn enc = encoder();
    if (!enc) return false;
    const cuuint64_t gdim[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t gstride[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), gdim, gstride, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A map depends only on (address, rows, K, box rows), so encoded maps are
// kept (a small table, most recent first) and reused: encoding costs more
// host time than a small contraction takes on the GPU.
bool make_map(CUtensorMap *map, const void *ptr, int rows, int K, int box_rows) {
    struct Entry {
        const void *ptr;
        int rows, K, box;
        CUtensorMap map;
    };
    static std::mutex mu;
    static std::vector<Entry> cache;
    std::lock_guard<std::mutex> lock(mu);
    for (size_t i = 0; i < cache.size(); ++i)
        if (cache[i].ptr == ptr && cache[i].rows == rows && cache[i].K == K && cache[i].box == box_rows) {
            *map = cache[i].map;
            return true;
        }
    Entry e{ptr, rows, K, box_rows, {}};
    if (!encode_map(&e.map, ptr, rows, K, box_rows)) return false;
    *map = e.map;
    if (cache.size() >= 512) cache.erase(cache.begin());
    cache.push_back(e);
    return true;
}

// Launch shape of one contraction. A CTA takes one 128-row weight tile and
// BN tokens; its loop costs a near-fixed time per 64-wide chunk (about 140
// cycles per MMA at M = 128, four MMAs a chunk), so the chunk count per CTA
// sets the time. The ring of one CTA fills an SM, so more CTAs than SMs run
// in two waves. Without a split the token tile is the smallest of 32, 64,
// 128 whose grid still fits one wave (more CTAs in flight at no extra chunks
// per CTA). A long reduction (K / 64 >= 64 chunks) is split, with token
// tiles of 128, into as many parts as fit one wave, at least 16 chunks each
// (measured at 128 tokens: 32-chunk splits 1.57 ms per prefill, 16-chunk
// 1.51, 8-chunk 1.54: shorter splits lose more to writing and re-reading the
// partial sums than they gain in parallel chunks).
struct GemmShape {
    int bn, S;
};

// A prompt of at most 32 tokens is one token tile: the weights' row tiles
// alone give too few CTAs to stream them at the memory's rate, so the
// reduction is split until the grid fills the SMs, with at least 4 chunks
// per split.
int small_splits(int tiles, int nk, int n_sm) {
    int S = n_sm / tiles;
    if (S > nk / 4) S = nk / 4;
    if (S > kMaxSplits) S = kMaxSplits;
    return S < 1 ? 1 : S;
}

GemmShape pick_shape(int M, int N, int K, int n_sm, bool norm) {
    const int rt = (M + 127) / 128, nk = K / 64;
    GemmShape g{128, 1};
    if (N <= 32) {
        g.bn = 32;
        g.S = small_splits(rt, nk, n_sm);
        if (norm && g.S < 2 && nk >= 2) g.S = 2;
        return g;
    }
    if (nk >= 64) {
        const int ctas = rt * ((N + 127) / 128);
        int S = n_sm / ctas;
        if (S > nk / 16) S = nk / 16;
        if (S > kMaxSplits) S = kMaxSplits;
        g.S = S < 1 ? 1 : S;
        if (norm && g.S < 2) g.S = 2;
        return g;
    }
    // a contraction that feeds an RMSNorm is split in any case (the pass
    // summing the parts also forms the norm): token tiles of 64 and as many
    // parts as fit one wave, at least 4 chunks each (the O-projection at 128
    // tokens: 4 parts of 8 chunks, 1.494 ms per prefill, against 2 parts of 16
    // with tiles of 32, 1.509, and 8 parts of 4 with tiles of 128, 1.527)
    if (norm && nk >= 8) {
        g.bn = 64;
        int S = n_sm / (rt * ((N + 63) / 64));
        if (S > nk / 4) S = nk / 4;
        if (S > kMaxSplits) S = kMaxSplits;
        g.S = S < 2 ? 2 : S;
        return g;
    }
    const int S = norm && nk >= 2 ? 2 : 1;
    for (int bn = 32; bn <= 128; bn *= 2)
        if (rt * ((N + bn - 1) / bn) * S <= n_sm || bn == 128) {
            g.bn = bn;
            break;
        }
    g.S = S;
    return g;
}

// keep_partials: with a K split the partial sums stay in part for the
// caller's own pass (no split-sum launch).
template <int BN, bool GATED = false>
cudaError_t launch_gemm_bn(const CUtensorMap *const *tas, const Segs &sg, const void *bhi, const void *blo, int N,
                           int K, float *part, int S, int *err, cudaStream_t s, const NormOut &nm = NormOut{},
                           bool keep_partials = false) {
    CUtensorMap th, tl;
    if (!make_map(&th, bhi, N, K, BN) || !make_map(&tl, blo, N, K, BN)) return cudaErrorInvalidValue;
    constexpr int smem = gemm_smem_bytes<BN>();
    static bool configured = false;
    if (!configured) {
        const cudaError_t e =
            cudaFuncSetAttribute(tc_gemm<BN, GATED>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    int tiles = 0;
    for (int i = 0; i < sg.n; ++i) tiles += sg.tiles[i];
    const dim3 grid(tiles, (N + BN - 1) / BN, S);
    const CUtensorMap &a0 = *tas[0], &a1 = GATED || sg.n > 1 ? *tas[1] : *tas[0], &a2 = sg.n > 2 ? *tas[2] : *tas[0];
    cudaError_t e =
        launch_pdl(tc_gemm<BN, GATED>, grid, dim3(kThreads), smem, s, a0, a1, a2, th, tl, sg, N, K, part, err);
    if (e != cudaSuccess || (S > 1 && keep_partials)) return e;
    const bool fused = nm.g && sg.M[0] <= kSnE * kSnThreads;
    if (S > 1 && fused)
        return launch_pdl(sum_splits_norm, dim3(N), dim3(kSnThreads), 0, s, part, S, N, sg.M[0], sg.Y[0], sg.ldy[0],
                          sg.R[0], nm.g, nm.eps, nm.hi, nm.lo);
    if (S > 1) e = launch_pdl(sum_splits, dim3(256), dim3(256), 0, s, part, S, N, sg.M[0], sg.Y[0], sg.ldy[0], sg.R[0]);
    if (e == cudaSuccess && nm.g)  // the norm on its own
        e = launch_pdl(norm_split, dim3(N), dim3(256), 0, s, sg.Y[0], sg.M[0], nm.g, nm.eps, nm.hi, nm.lo);
    return e;
}

template <int BN>
cudaError_t launch_one(const CUtensorMap &ta, const void *bhi, const void *blo, int M, int N, int K, float *Y, int ldy,
                       const float *R, float *part, int S, int *err, cudaStream_t s, const NormOut &nm) {
    Segs sg{};
    sg.n = 1;
    sg.tiles[0] = (M + 127) / 128;
    sg.M[0] = M;
    sg.Y[0] = Y;
    sg.ldy[0] = ldy;
    sg.R[0] = R;
    sg.mtot = M;
    const CUtensorMap *tas[1] = {&ta};
    return launch_gemm_bn<BN>(tas, sg, bhi, blo, N, K, part, S, err, s, nm);
}

}  // namespace

bool encode_weight_map(CUtensorMap *map, const void *w, int rows, int K) { return make_map(map, w, rows, K, 128); }

bool encode_gated_map(CUtensorMap *map, const void *w, int rows, int K) { return make_map(map, w, rows, K, 64); }

size_t gemm_workspace_floats(int M, int N, int K, int n_sm, bool norm) {
    const GemmShape g = pick_shape(M, N, K, n_sm, norm);
    return g.S > 1 ? (size_t)g.S * N * M : 0;
}

cudaError_t gemm(const CUtensorMap &wmap, const void *bhi, const void *blo, int M, int N, int K, float *Y, int ldy,
                 const float *R, float *work, size_t work_floats, int *err, int n_sm, cudaStream_t s,
                 const NormOut &nm) {
    if (K % 64 || M < 1 || N < 1 || (nm.g && ldy != M)) return cudaErrorInvalidValue;
    const GemmShape g = pick_shape(M, N, K, n_sm, nm.g != nullptr);
    const int S = (size_t)g.S * N * M > work_floats ? 1 : g.S;  // no room for the partials: one pass
    switch (g.bn) {
        case 128: return launch_one<128>(wmap, bhi, blo, M, N, K, Y, ldy, R, work, S, err, s, nm);
        case 64: return launch_one<64>(wmap, bhi, blo, M, N, K, Y, ldy, R, work, S, err, s, nm);
        default: return launch_one<32>(wmap, bhi, blo, M, N, K, Y, ldy, R, work, S, err, s, nm);
    }
}

cudaError_t gemm_multi(int nseg, const CUtensorMap *const *maps, const int *M, float *const *Y, const int *ldy,
                       const void *bhi, const void *blo, int N, int K, int *err, int n_sm, cudaStream_t s, float *work,
                       size_t work_floats, int *S_used) {
    *S_used = 1;
    if (K % 64 || N < 1 || nseg < 1 || nseg > 3) return cudaErrorInvalidValue;
    Segs sg{};
    sg.n = nseg;
    int tiles = 0;
    for (int i = 0; i < nseg; ++i) {
        if (M[i] < 1) return cudaErrorInvalidValue;
        sg.tiles[i] = (M[i] + 127) / 128;
        sg.M[i] = M[i];
        sg.Y[i] = Y[i];
        sg.ldy[i] = ldy[i];
        sg.R[i] = nullptr;
        sg.off[i] = sg.mtot;
        sg.mtot += M[i];
        tiles += sg.tiles[i];
    }
    if (N <= 32) {
        int S = small_splits(tiles, K / 64, n_sm);
        if ((size_t)S * N * sg.mtot > work_floats) S = 1;
        *S_used = S;
        return launch_gemm_bn<32>(maps, sg, bhi, blo, N, K, work, S, err, s, NormOut{}, true);
    }
    // the smallest token tile whose grid fits one wave (as pick_shape)
    int bn = 128;
    for (int b = 32; b < 128; b *= 2)
        if (tiles * ((N + b - 1) / b) <= n_sm) {
            bn = b;
            break;
        }
    switch (bn) {
        case 32: return launch_gemm_bn<32>(maps, sg, bhi, blo, N, K, nullptr, 1, err, s);
        case 64: return launch_gemm_bn<64>(maps, sg, bhi, blo, N, K, nullptr, 1, err, s);
        default: return launch_gemm_bn<128>(maps, sg, bhi, blo, N, K, nullptr, 1, err, s);
    }
}

size_t gemm_multi_workspace_floats(int nseg, const int *M, int N, int K, int n_sm) {
    if (N > 32) return 0;
    int tiles = 0, mtot = 0;
    for (int i = 0; i < nseg; ++i) {
        tiles += (M[i] + 127) / 128;
        mtot += M[i];
    }
    return (size_t)small_splits(tiles, K / 64, n_sm) * N * mtot;
}

cudaError_t gemm_gated(const CUtensorMap &wg, const CUtensorMap &wu, int F, const void *bhi, const void *blo, int N,
                       int K, uint16_t *hhi, uint16_t *hlo, int *err, int n_sm, cudaStream_t s) {
    if (K % 64 || N < 1 || F < 1) return cudaErrorInvalidValue;
    Segs sg{};
    sg.n = 1;
    sg.tiles[0] = (F + 63) / 64;
    sg.M[0] = F;
    sg.ldy[0] = F;
    sg.mtot = F;
    sg.hhi = hhi;
    sg.hlo = hlo;
    const CUtensorMap *maps[2] = {&wg, &wu};
    int bn = 128;
    for (int b = 32; b < 128; b *= 2)
        if (sg.tiles[0] * ((N + b - 1) / b) <= n_sm) {
            bn = b;
            break;
        }
    switch (bn) {
        case 32: return launch_gemm_bn<32, true>(maps, sg, bhi, blo, N, K, nullptr, 1, err, s);
        case 64: return launch_gemm_bn<64, true>(maps, sg, bhi, blo, N, K, nullptr, 1, err, s);
        default: return launch_gemm_bn<128, true>(maps, sg, bhi, blo, N, K, nullptr, 1, err, s);
    }
}

cudaError_t run(const Model &m, const Scratch &sc, const int32_t *d_tokens, int n, int pos0, float *out_logits,
                int32_t *out_token, cudaStream_t s) {
    const int d = m.d, Hq = m.Hq, Hkv = m.Hkv, hd = m.hd, F = m.F, qd = Hq * hd, kvd = Hkv * hd;
    const int qkv = qd + 2 * kvd;
    cudaError_t e = cudaSuccess;
    auto ok = [&](cudaError_t x) {
        if (e == cudaSuccess) e = x;
        return e == cudaSuccess;
    };
    ok(launch_pdl(embed_rows, dim3(n), dim3(256), 0, s, m.embed, d_tokens, n, d, m.V, sc.X, sc.err));
    for (int l = 0; l < m.L && e == cudaSuccess; ++l) {
        const LayerMaps &lm = m.maps[l];
        const size_t kv_off = (size_t)l * m.kv_layer_stride;
        // attention block
        // (later layers: the previous down projection's split sum formed the norm)
        if (l == 0)
            ok(launch_pdl(norm_split, dim3(n), dim3(256), 0, s, sc.X, d, m.attn_norm[0], m.eps, sc.Ahi, sc.Alo));
        {  // q, k and v in one launch
            const CUtensorMap *maps[3] = {&lm.wq, &lm.wk, &lm.wv};
            const int Ms[3] = {qd, kvd, kvd}, lds[3] = {qkv, qkv, qkv};
            float *Ys[3] = {sc.QKV, sc.QKV + qd, sc.QKV + qd + kvd};
            int Sq = 1;
            ok(gemm_multi(3, maps, Ms, Ys, lds, sc.Ahi, sc.Alo, n, d, sc.err, m.n_sm, s, sc.work, sc.work_floats,
                          &Sq));
            // RoPE and the KV append (a short prompt: from the split partial sums)
            const int per_tok = n >= 64 ? 1 : std::min(8, (64 + n - 1) / n);
            ok(launch_pdl(rope_append, dim3(n, per_tok), dim3(256), 0, s, sc.QKV, Sq > 1 ? sc.work : nullptr,
                          Sq > 1 ? Sq : 0, n, Hq, Hkv, hd, pos0, m.rope, m.max_seq, m.kc + kv_off, m.vc + kv_off));
        }
        {  // causal attention on the tensor cores (every supported group size: G <= kFaRows)
            const int QB = kFaRows / (Hq / Hkv);
            const dim3 grid(Hkv, (n + QB - 1) / QB);
            if (hd == 64)
                ok(launch_pdl(attend_prefill_mma<64>, grid, dim3(kFaWarps * 32), 0, s, sc.QKV, n, Hq, Hkv, pos0,
                              m.max_seq, m.kc + kv_off, m.vc + kv_off, sc.Ahi, sc.Alo));
            else
                ok(launch_pdl(attend_prefill_mma<128>, grid, dim3(kFaWarps * 32), 0, s, sc.QKV, n, Hq, Hkv, pos0,
                              m.max_seq, m.kc + kv_off, m.vc + kv_off, sc.Ahi, sc.Alo));
        }
        // O-projection + residual, then the MLP's RMSNorm
        ok(gemm(lm.wo, sc.Ahi, sc.Alo, d, n, qd, sc.X, d, sc.X, sc.work, sc.work_floats, sc.err, m.n_sm, s,
                NormOut{m.mlp_norm[l], m.eps, sc.Ahi, sc.Alo}));
        // gate and up in one launch, h = silu(g) * u formed in its epilogue
        ok(gemm_gated(lm.wg, lm.wu, F, sc.Ahi, sc.Alo, n, d, sc.Hhi, sc.Hlo, sc.err, m.n_sm, s));
        // down projection + residual, then the next layer's attention RMSNorm
        const NormOut next = l + 1 < m.L ? NormOut{m.attn_norm[l + 1], m.eps, sc.Ahi, sc.Alo} : NormOut{};
        ok(gemm(lm.wd, sc.Hhi, sc.Hlo, d, n, F, sc.X, d, sc.X, sc.work, sc.work_floats, sc.err, m.n_sm, s, next));
    }
    if (e != cudaSuccess) return e;
    // LM head of the last prompt position
    const int blocks = 2 * m.n_sm;
    if (!ok(launch_pdl(lm_head_rows, dim3(blocks), dim3(512), sizeof(float) * d, s, sc.X + (size_t)(n - 1) * d,
                       m.final_norm, m.eps, m.embed, m.V, d, out_logits, sc.keys)))
        return e;
    ok(launch_pdl(argmax_keys, dim3(1), dim3(256), 0, s, sc.keys, blocks, out_token));
    return e;
}

}  // namespace mkpf

// Unit entry of the tensor-core contraction (tests and measurement).
extern "C" int mk_tc_gemm(const void *d_w, int32_t M, int32_t K, const void *d_bhi, const void *d_blo, int32_t N,
                          float *d_y, const float *d_r, int32_t *d_status, void *stream) {
    if (!d_w || !d_bhi || !d_blo || !d_y || !d_status || M < 1 || N < 1 || K < 64 || K % 64) return -1;
    if ((reinterpret_cast<uintptr_t>(d_w) | reinterpret_cast<uintptr_t>(d_bhi) | reinterpret_cast<uintptr_t>(d_blo)) & 15u)
        return -1;
    CUtensorMap wm;
    if (!mkpf::encode_weight_map(&wm, d_w, M, K)) return -4;
    int dev = 0, n_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return -2;
    // the K-split partials of this entry live in a workspace it keeps (grown
    // when a larger contraction needs more; freed at exit)
    static float *work = nullptr;
    static size_t work_floats = 0;
    const size_t need = mkpf::gemm_workspace_floats(M, N, K, n_sm, false);
    if (need > work_floats) {
        if (work) {
            cudaDeviceSynchronize();
            cudaFree(work);
        }
        work = nullptr;
        work_floats = 0;
        if (cudaMalloc(&work, need * sizeof(float)) == cudaSuccess) work_floats = need;
    }
    const cudaError_t e = mkpf::gemm(wm, d_bhi, d_blo, M, N, K, d_y, M, d_r, work, work_floats, d_status, n_sm,
                                     static_cast<cudaStream_t>(stream), mkpf::NormOut{});
    return e == cudaSuccess ? 0 : -2;
}
