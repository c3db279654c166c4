#pragma once
// mk_kernel.cuh — the persistent decode megakernel (sm_103a), device code.
// Included by mk_kernel_hd64.cu and mk_kernel_hd128.cu, which instantiate it.
//
// One CTA per SM interprets that SM's instruction queue (planned on the host,
// see mk_host.cpp). The design is the one described in "Revolution der
// KI-Beschleunigung: Wie ein Low-Latency Megakernel den Llama-1B Turbo
// zündet" (dasgeld.co), rebuilt for GB300:
//   * the whole decode step is one launch; stages that used to be separate
//     kernels are instructions (megakernel paragraphs);
//   * every instruction waits for exactly the data it consumes through flags
//     in global memory (synchronisation paragraph): each activation element
//     is a tagged 8-byte word {value, step/version tag}; consumers poll the
//     words they read, so an edge costs one round trip and producers never
//     wait for write acknowledgements;
//   * shared memory is a ring of pages: a producer warp streams the next
//     instructions' weights (and cached keys/values) into free pages with
//     cp.async.bulk while the consumer warps compute, across dependency
//     waits, so HBM keeps streaming during synchronisation (shared-memory
//     paging paragraph);
//   * bf16 weights, fp32 accumulation (latency paragraph).
//
// CTA layout: warps 0..7 are consumers (GEMV / attention math), warp 8 is
// the producer: its lane 0 waits for pages and arms their barriers, its
// lanes issue the bulk copies. Page p has a "full" mbarrier
// (producer -> consumers, completed by the copy's transaction bytes) and an
// "empty" mbarrier (8 consumer warps -> producer).
//
// Every wait is bounded (%globaltimer): on expiry the CTA records a timeout
// in the status word, raises the abort flag that all CTAs poll, waits for
// its own copies in flight and returns. Nothing traps. Counters remain only
// for the LM head's global argmax and for the end of the step.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mk_plan.h"

namespace mk {

extern __shared__ __align__(1024) uint8_t mk_smem[];

// Everything below has internal linkage: each instance translation unit
// carries its own copy.
namespace {

// ---------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Bulk (non-tensor) copy global -> this CTA's shared memory, completing
// `bytes` transaction bytes on `bar`. 16-byte aligned addresses and size.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add(uint32_t *p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t atom_acq_rel_add(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(p), "r"(v)
                 : "memory");
    return old;
}

__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

// Consumer barrier that also returns whether any consumer thread passed
// `pred` = true, so failure decisions stay uniform across the warps.
__device__ __forceinline__ bool consumer_sync_any(bool pred) {
    uint32_t cnt;
    asm volatile(
        "{\n\t.reg .pred q;\n\t"
        "setp.ne.u32 q, %2, 0;\n\t"
        "bar.red.popc.u32 %0, 1, %1, q;\n\t}"
        : "=r"(cnt)
        : "n"(kConsumerThreads), "r"((uint32_t)pred)
        : "memory");
    return cnt != 0;
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

// fp32 -> bf16, round to nearest even (finite inputs; NaN kept quiet).
__device__ __forceinline__ uint16_t f2bf(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7F800000u) == 0x7F800000u) return uint16_t((u >> 16) | ((u & 0xFFFFu) ? 0x40u : 0u));
    u += 0x7FFFu + ((u >> 16) & 1u);
    return uint16_t(u >> 16);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

__device__ __forceinline__ float ldcg(const float *p) { return __ldcg(p); }

// ---------------------------------------------------------------------------
// Address self-checks. A build with MK_CHECKED validates every global access
// against the byte ranges the host registered (weights, caches, scratch,
// outputs) and every computed shared-memory access against the CTA's
// allocation; the first violation is recorded in p.dbg and the access is
// skipped. Without MK_CHECKED the checks compile to `true`.
// ---------------------------------------------------------------------------

#ifdef MK_CHECKED
__device__ __noinline__ void chk_record(const Params &p, int site, uintptr_t a, size_t bytes) {
    if (p.dbg && atomicCAS(p.dbg, 0ull, (unsigned long long)site) == 0ull) {
        p.dbg[1] = a;
        p.dbg[2] = bytes;
        p.dbg[3] = ((unsigned long long)blockIdx.x << 32) | threadIdx.x;
        __threadfence();
    }
}
__device__ __noinline__ bool chk_global(const Params &p, const void *ptr, size_t bytes, int site) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(ptr);
    for (int i = 0; i < p.n_ranges; ++i)
        if (a >= p.ranges[2 * i] && a + bytes <= p.ranges[2 * i + 1]) return true;
    if (p.out_logits && a >= (uintptr_t)p.out_logits && a + bytes <= (uintptr_t)(p.out_logits + p.V))
        return true;
    if (p.out_token && a >= (uintptr_t)p.out_token && a + bytes <= (uintptr_t)(p.out_token + 1))
        return true;
    if (p.d_token && a >= (uintptr_t)p.d_token && a + bytes <= (uintptr_t)(p.d_token + 1))
        return true;
    if (p.trace && a >= (uintptr_t)p.trace &&
        a + bytes <= (uintptr_t)(p.trace + (size_t)gridDim.x * p.trace_cap * kTraceWords))
        return true;
    chk_record(p, site, a, bytes);
    return false;
}
__device__ __noinline__ bool chk_shared(const Params &p, const void *ptr, size_t bytes, int site) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(ptr), b = reinterpret_cast<uintptr_t>(mk_smem);
    if (__isShared(ptr) && a >= b && a + bytes <= b + kSmemBytes) return true;
    chk_record(p, site, a, bytes);
    return false;
}
#define CHK(ptr, bytes, site) chk_global(p, (ptr), (bytes), (site))
#define CHKS(ptr, bytes, site) chk_shared(p, (ptr), (bytes), (site))
#else
#define CHK(ptr, bytes, site) true
#define CHKS(ptr, bytes, site) true
#endif

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw: "Parallel random numbers: as
// easy as 1, 2, 3", SC'11): word 0 of the output block for counter (c0..c3)
// and key (k0, k1). Ten rounds of two 32x32->64 multiplies by M0, M1 with
// the key bumped by the Weyl constants W0, W1 after every round.
__device__ __forceinline__ uint32_t philox_w0(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                              uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
        c0 = hi1 ^ c1 ^ k0;
        c1 = lo1;
        c2 = hi0 ^ c3 ^ k1;
        c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c0;
}

// Uniform in the open interval (0, 1) from one 32-bit word: the top 23 bits
// plus 1/2, over 2^23. Every step is exact in fp32 (the largest value is
// 1 - 2^-24), so -log(u) is never 0 and the noise below stays finite for
// every word, the all-ones word included.
__device__ __forceinline__ float gumbel_from_word(uint32_t x) {
    const float u = ((float)(x >> 9) + 0.5f) * (1.0f / 8388608.0f);
    return -logf(-logf(u));
}

// Gumbel noise of vocabulary entry i for the sequence on KV slot `slot` at
// position `pos`: g = -log(-log(u)), u from word 0 of Philox(i, pos, slot, 0;
// seed). argmax_i(z_i + g_i) is a draw from softmax(z).
__device__ __forceinline__ float gumbel_noise(uint32_t i, int pos, int slot, uint32_t seed_lo, uint32_t seed_hi) {
    return gumbel_from_word(philox_w0(i, (uint32_t)pos, (uint32_t)slot, 0u, seed_lo, seed_hi));
}

// Orderable key for the argmax: larger value wins, then lower index.
__device__ __forceinline__ unsigned long long argmax_key(float v, uint32_t idx) {
    uint32_t u = __float_as_uint(v);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return (static_cast<unsigned long long>(u) << 32) | (0xFFFFFFFFu - idx);
}

// ---------------------------------------------------------------------------
// Tagged activation words. Every activation element lives in global memory as
// {float bits, tag} and is written with ONE relaxed 8-byte store, read with
// relaxed 8-byte (or paired 8-byte) loads; each 8-byte access is single-copy
// atomic, so a reader that sees the expected tag sees the value written with
// it. The tag is (step epoch << 8) | version, so data of an
// earlier step, or an earlier version of the in-place residual stream, never
// matches. A consumer therefore needs no counter and no separate acquire:
// polling the words it consumes is its dependency wait, and a producer never
// waits for its writes to be acknowledged.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ll_store(uint2 *dst, float v, uint32_t tag) {
    const unsigned long long w =
        ((unsigned long long)tag << 32) | (unsigned long long)__float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(dst), "l"(w) : "memory");
}

// Two tagged elements; each 64-bit half is read single-copy atomically.
__device__ __forceinline__ uint4 ll_ld16(const uint2 *src) {
    unsigned long long a, b;
    asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(src) : "memory");
    return make_uint4((uint32_t)a, (uint32_t)(a >> 32), (uint32_t)b, (uint32_t)(b >> 32));
}

__device__ __forceinline__ uint2 ll_ld8(const uint2 *src) {  // one tagged element
    unsigned long long a;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(a) : "l"(src) : "memory");
    return make_uint2((uint32_t)a, (uint32_t)(a >> 32));
}

// Batched steps keep x, the attention output and h as plain fp32 with the
// kMaxBatch sequence slots interleaved, so that the batched GEMV's input
// reads are coalesced: element e of sequence b sits in group (e/32)*2 +
// (e/4)%2 of 128 floats, at b*16 + ((e/8)%4)*4 + e%4. The 32 lanes (b, t) of
// a warp that read elements 8t .. 8t+3 (or 8t+4 .. 8t+7) of a 32-element
// block of every sequence then read one contiguous 512-byte span. These
// buffers are published by completion counters (release by the producing
// instruction, acquire before the consuming one), not by tags.
__device__ __forceinline__ size_t bofs(int b, int e) {
    return (size_t)(((e >> 5) * 2 + ((e >> 2) & 1)) * 128 + b * 16 + ((e >> 3) & 3) * 4 + (e & 3));
}

__device__ __forceinline__ float4 ld_relaxed_f4(const float *src) {
    float4 v;
    asm volatile("ld.relaxed.gpu.global.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(src)
                 : "memory");
    return v;
}

__device__ __forceinline__ float ld_relaxed_f(const float *src) {
    float v;
    asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(src) : "memory");
    return v;
}

// ---------------------------------------------------------------------------
// Shared state
// ---------------------------------------------------------------------------
struct Misc {
    float red8[kConsumerWarps];
    unsigned long long best8[kConsumerWarps];
    volatile int32_t flag;      // broadcast slot
    volatile int32_t polling;   // consumers are polling for an input (producer throttles)
    volatile int32_t aborted;   // this CTA gave up
    volatile uint32_t n_issued; // tiles issued by the producer
    uint32_t ep8;               // this step's epoch << 8
    int32_t staged_key;         // (op << 16 | layer) whose input xbuf holds, -1 none
    float staged_ss;            // its sum of squares
    int32_t gcount;             // filtered draw: candidates gathered
    long long phase[3];         // trace: intra-instruction phase stamps
    long long tile_wait;        // trace: ns thread 0 spent waiting for tiles to land
};

struct Ctx {
    uint8_t *pages;
    float *xbuf;
    float *red;
    float *resid;
    float *dred;
    uint64_t *full, *empty;
    Misc *misc;
};

// Bounded spinning: every 16th call checks the abort flag and the clock; on
// expiry it records a timeout, raises the abort flag and tells the caller to
// give up.
struct Spin {
    uint64_t t0 = 0;
    uint32_t it = 0;
    __device__ __forceinline__ bool keep_going(const Params &p) {
        if ((++it & 15u) != 0) return true;
        if (*(volatile int32_t *)p.abort_flag) return false;
        const uint64_t now = gtimer();
        if (t0 == 0) {
            t0 = now;
            return true;
        }
        if (now - t0 > p.timeout_ns) {
            atomicCAS(p.status, DS_OK, DS_TIMEOUT);
            atomicExch(p.abort_flag, 1);
            return false;
        }
        return true;
    }
};

// Waits for one tagged element. Returns false on abort/timeout.
__device__ __forceinline__ bool ll_read1(const Params &p, const uint2 *src, uint32_t tag, float &out) {
    if (!CHK(src, 8, 37)) return false;
    Spin sp;
    while (true) {
        const uint2 v = ll_ld8(src);
        if (v.y == tag) {
            out = __uint_as_float(v.x);
            return true;
        }
        if (!sp.keep_going(p)) return false;
    }
}

// Waits for N independent tagged elements (any addresses), all loads of a
// poll in flight together. Returns false on abort/timeout.
template <int N>
__device__ __forceinline__ bool ll_read_n(const Params &p, const uint2 *const *src, uint32_t tag,
                                          float *out) {
#pragma unroll
    for (int k = 0; k < N; ++k)
        if (!CHK(src[k], 8, 37)) return false;
    Spin sp;
    while (true) {
        uint2 v[N];
#pragma unroll
        for (int k = 0; k < N; ++k) v[k] = ll_ld8(src[k]);
        bool ok = true;
#pragma unroll
        for (int k = 0; k < N; ++k) ok = ok && v[k].y == tag;
        if (ok) {
#pragma unroll
            for (int k = 0; k < N; ++k) out[k] = __uint_as_float(v[k].x);
            return true;
        }
        if (!sp.keep_going(p)) return false;
    }
}

// Bounded wait on an mbarrier phase.
__device__ bool wait_bar(const Params &p, uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    Spin sp;
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (!sp.keep_going(p)) return false;
    }
}

// Consumer wait for page pg to be full in the phase of parity par; on traced
// steps thread 0 adds the time it waited to the instruction's tile_wait.
__device__ __forceinline__ bool wait_tile(const Params &p, const Ctx &cx, int pg, uint32_t par,
                                          bool tracing) {
    if (!tracing) return wait_bar(p, &cx.full[pg], par);
    uint64_t t0 = 0;
    if (threadIdx.x == 0) t0 = gtimer();
    const bool ok = wait_bar(p, &cx.full[pg], par);
    if (threadIdx.x == 0) cx.misc->tile_wait += (long long)(gtimer() - t0);
    return ok;
}

// Trace stamp of an intra-instruction phase (thread 0, traced steps only).
__device__ __forceinline__ void phase_stamp(const Params &p, const Ctx &cx, int k) {
    if (p.trace && threadIdx.x == 0) cx.misc->phase[k] = (long long)gtimer();
}

// Pulls the 64-byte record of instruction i into L1 ahead of its load_instr.
__device__ __forceinline__ void prefetch_instr(const Params &p, int i) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p.instr + i));
}

__device__ __forceinline__ Instr load_instr(const Params &p, int i) {
    Instr in;
    if (!CHK(p.instr + i, sizeof(Instr), 1)) {
        memset(&in, 0, sizeof in);
        in.wait_ctr = -1;
        in.op = OP_QKV;
        return in;
    }
    const int4 *src = reinterpret_cast<const int4 *>(p.instr + i);
    int4 *dst = reinterpret_cast<int4 *>(&in);
#pragma unroll
    for (int k = 0; k < 4; ++k) dst[k] = __ldg(src + k);
    return in;
}

__device__ __forceinline__ const Geo &geo_of(const Params &p, int op) {
    switch (op) {
        case OP_QKV: return p.geo_qkv;
        case OP_OPROJ: return p.geo_o;
        case OP_GATEUP: return p.geo_gu;
        case OP_DOWN: return p.geo_down;
        default: return p.geo_lm;
    }
}

__device__ __forceinline__ int current_token(const Params &p, int b = 0) {
    if (p.d_token && !CHK(p.d_token + b, 4, 33)) return -1;
    return p.d_token ? *(volatile const int32_t *)(p.d_token + b) : p.token;
}

// Sequence of an instruction in a batched step (attention instructions carry
// it in `mat`), its position and its KV-cache slot.
__device__ __forceinline__ int seq_of(const Params &p, const Instr &in) { return p.nb > 1 ? in.mat : 0; }
__device__ __forceinline__ int pos_of(const Params &p, int b) { return p.nb > 1 ? p.posb[b] : p.pos; }
__device__ __forceinline__ int slot_of(const Params &p, int b) { return p.nb > 1 ? b : p.bslot; }

// ---------------------------------------------------------------------------
// Attention split bookkeeping (identical on producer and consumer side).
// Cached positions [0, pos) are cut into seff <= S contiguous chunks of at
// least one tile; the last active split also owns the new position `pos`
// and merges the splits.
// ---------------------------------------------------------------------------
struct AttnRange {
    int active, t0, t1, has_new;
};

__device__ __forceinline__ int attn_seff(const Params &p, int pos) {
    const int per = p.ppt * kMinSplitTiles;
    int need = (pos + per - 1) / per;
    if (need < 1) need = 1;
    return need < p.S ? need : p.S;
}

__device__ __forceinline__ AttnRange attn_range(const Params &p, int split, int pos) {
    AttnRange r;
    const int seff = attn_seff(p, pos);
    r.active = split < seff;
    const int chunk = (pos + seff - 1) / seff;
    r.t0 = split * chunk;
    if (r.t0 > pos) r.t0 = pos;
    r.t1 = r.t0 + chunk;
    if (r.t1 > pos) r.t1 = pos;
    r.has_new = (split == seff - 1);
    return r;
}

__device__ __forceinline__ int num_tiles(const Params &p, const Instr &in) {
    if (in.op == OP_ATTN) {
        const AttnRange r = attn_range(p, in.a1, pos_of(p, seq_of(p, in)));
        if (!r.active) return 0;
        return (r.t1 - r.t0 + p.ppt - 1) / p.ppt;
    }
    const Geo &g = geo_of(p, in.op);
    const int per = (in.op == OP_GATEUP) ? g.rt / 2 : g.rt;
    const int nrb = (in.a1 + per - 1) / per;
    return p.nb > 1 ? nrb * (g.K / g.pad) : nrb;  // batched: one tile per (K-chunk, row block)
}

// ---------------------------------------------------------------------------
// Tile copies: tile j of an instruction is one or two contiguous global
// ranges copied into one page.
// ---------------------------------------------------------------------------
struct TileCopy {
    const void *src0, *src1;
    uint32_t bytes0, bytes1;  // bytes1 == 0: single copy
    uint32_t dst1;            // page offset of the second copy
};

__device__ __forceinline__ TileCopy tile_copy(const Params &p, const Instr &in, int j) {
    TileCopy c;
    c.src1 = nullptr;
    c.bytes1 = 0;
    c.dst1 = 0;
    if (in.op == OP_ATTN) {
        const int b = seq_of(p, in);
        const AttnRange r = attn_range(p, in.a1, pos_of(p, b));
        const int ts = r.t0 + j * p.ppt;
        int n = r.t1 - ts;
        if (n > p.ppt) n = p.ppt;
        const size_t base = (((size_t)in.layer * p.max_batch + slot_of(p, b)) * p.Hkv + in.a0) * p.max_seq * p.hd +
                            (size_t)ts * p.hd;
        c.bytes0 = c.bytes1 = (uint32_t)n * p.hd * 2;
        c.src0 = p.kc + base;
        c.src1 = p.vc + base;
        c.dst1 = kPageBytes / 2;
        return c;
    }
    const Geo &g = geo_of(p, in.op);
    const int per = (in.op == OP_GATEUP) ? g.rt / 2 : g.rt;
    int rows = in.a1 - j * per;
    if (rows > per) rows = per;
    const size_t row0 = (size_t)in.a0 + (size_t)j * per;
    const LayerW *lw = p.layers + in.layer;
    c.bytes0 = (uint32_t)rows * g.K * 2;
    switch (in.op) {
        case OP_GATEUP:
            c.src0 = lw->w_gate + row0 * g.K;
            c.src1 = lw->w_up + row0 * g.K;
            c.bytes1 = c.bytes0;
            c.dst1 = (uint32_t)per * g.K * 2;
            break;
        case OP_QKV: {
            // rows of the stacked [Wq; Wk; Wv]; a tile crosses at most one boundary
            const size_t qd = (size_t)p.Hq * p.hd, kvd = (size_t)p.Hkv * p.hd;
            const size_t end = row0 + (size_t)rows;
            const int m0 = row0 < qd ? 0 : (row0 < qd + kvd ? 1 : 2);
            const size_t start0 = m0 == 0 ? 0 : (m0 == 1 ? qd : qd + kvd);
            const size_t bound = m0 == 0 ? qd : (m0 == 1 ? qd + kvd : qd + 2 * kvd);
            const uint16_t *mats[3] = {lw->wq, lw->wk, lw->wv};
            c.src0 = mats[m0] + (row0 - start0) * g.K;
            if (end > bound && m0 < 2) {
                c.bytes0 = (uint32_t)((bound - row0) * g.K * 2);
                c.src1 = mats[m0 + 1];
                c.bytes1 = (uint32_t)((end - bound) * g.K * 2);
                c.dst1 = c.bytes0;
            }
            break;
        }
        case OP_OPROJ: c.src0 = lw->wo + row0 * g.K; break;
        case OP_DOWN: c.src0 = lw->w_down + row0 * g.K; break;
        default: c.src0 = p.lm_w + row0 * g.K; break;
    }
    return c;
}

__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Second walk over the queue, ahead of the ring: tiles the ring cannot hold
// yet are pulled into L2 while the producer would otherwise wait for a free
// page, so HBM keeps streaming through dependency waits and the tiles of the
// next instructions later land from L2.
struct L2Cursor {
    int i, j, nt;  // instruction, tile within it, its tile count
    uint32_t t;    // global tile index of (i, j)
};

__device__ __forceinline__ void l2_advance(const Params &p, L2Cursor &c, int qe) {
    ++c.t;
    if (++c.j < c.nt) return;
    c.j = 0;
    c.nt = 0;
    while (++c.i < qe && (c.nt = num_tiles(p, load_instr(p, c.i))) == 0) {
    }
}

__device__ __forceinline__ void l2_prefetch_tile(const Params &p, const L2Cursor &c) {
    const TileCopy tc = tile_copy(p, load_instr(p, c.i), c.j);
    if (CHK(tc.src0, tc.bytes0, 35)) prefetch_l2(tc.src0, tc.bytes0);
    if (tc.bytes1 && CHK(tc.src1, tc.bytes1, 36)) prefetch_l2(tc.src1, tc.bytes1);
}

// ---------------------------------------------------------------------------
// Producer: walks the same queue as the consumers and issues every tile into
// the page ring. Per instruction it resolves the tile sources once; per tile
// it only advances pointers (GEMV tiles of one instruction are equally
// strided rows of one or two matrices).
// ---------------------------------------------------------------------------
// Accumulators of a batched instruction (kBatchAcc floats): per output row
// (two per row for gate/up) and sequence, for the whole instruction, or a
// ring of 8 tiles.
__device__ __forceinline__ bool batch_ring(int n, int op) {
    return n * (op == OP_GATEUP ? 2 : 1) * kMaxBatch > kBatchAcc;
}

// Tile j of a batched instruction: (K-chunk, row block), in groups of gsz
// row blocks (all K-chunks of a group before the next group).
struct BTile {
    int kc, rb;
};
__device__ __forceinline__ BTile batch_tile(int j, int nrb, int nkc, int gsz) {
    const int grp = j / (gsz * nkc);
    const int q = j - grp * gsz * nkc;
    const int left = nrb - grp * gsz;
    const int gs = left < gsz ? left : gsz;
    return {q / gs, grp * gsz + q % gs};
}

// Start of weight row `row` (stacked [Wq; Wk; Wv] rows for QKV; for gate/up
// `up` selects the up matrix) of a batched GEMV instruction.
__device__ __forceinline__ const uint16_t *batch_row(const Params &p, const Instr &in, size_t row, bool up) {
    const LayerW *lw = p.layers + in.layer;
    const size_t K = (size_t)geo_of(p, in.op).K;
    switch (in.op) {
        case OP_QKV: {
            const size_t qd = (size_t)p.Hq * p.hd, kvd = (size_t)p.Hkv * p.hd;
            if (row < qd) return lw->wq + row * K;
            if (row < qd + kvd) return lw->wk + (row - qd) * K;
            return lw->wv + (row - qd - kvd) * K;
        }
        case OP_GATEUP: return (up ? lw->w_up : lw->w_gate) + row * K;
        case OP_OPROJ: return lw->wo + row * K;
        case OP_DOWN: return lw->w_down + row * K;
        default: return p.lm_w + row * K;
    }
}

// Runs on all 32 lanes of the producer warp: lane 0 waits for free pages
// and arms each page's barrier, the lanes share a tile's copies.
__device__ void producer(const Params &p, const Ctx &cx, int qb, int qe) {
    const int lane = threadIdx.x & 31;
    const uint64_t pol = policy_evict_first();
    uint32_t t = 0;
    int pg = 0;         // page of tile t
    uint32_t use = 0;   // how many times page pg has been filled before (parity of its phase)
    const uint32_t back = (uint32_t)p.max_inflight, pback = (uint32_t)p.poll_inflight;
    const uint32_t la = p.nb > 1 ? 0u : (uint32_t)p.l2_tiles;  // tiles beyond the ring pulled into L2
    L2Cursor lc{qb, 0, qb < qe ? num_tiles(p, load_instr(p, qb)) : 0, 0u};
    if (lc.nt == 0 && qb < qe) {
        lc.j = -1;
        l2_advance(p, lc, qe);
        lc.t = 0;
    }
    for (int i = qb; i < qe; ++i) {
        const Instr in = load_instr(p, i);
        if (i + 1 < qe) prefetch_instr(p, i + 1);
        const int nt = num_tiles(p, in);
        // batched steps: tile j = (K-chunk, row block) in the consumers' order
        const bool batched = p.nb > 1 && in.op != OP_ATTN;
        int nrb = 1, nkc = 1, KC = 0, bper = 0, gsz = 1;
        if (batched) {
            const Geo &g = geo_of(p, in.op);
            KC = g.pad;
            nkc = g.K / KC;
            bper = in.op == OP_GATEUP ? g.rt / 2 : g.rt;
            nrb = (in.a1 + bper - 1) / bper;
            gsz = batch_ring(in.a1, in.op) ? 8 : nrb;
        }
        // GEMV ops other than the stacked QKV: tile j = tile 0 shifted by j*per rows
        const bool strided = !batched && (in.op == OP_OPROJ || in.op == OP_GATEUP || in.op == OP_DOWN || in.op == OP_LMHEAD);
        TileCopy c0{};
        size_t row_bytes = 0;
        int per = 0;
        if (strided && nt > 0) {
            c0 = tile_copy(p, in, 0);
            const Geo &g = geo_of(p, in.op);
            row_bytes = (size_t)g.K * 2;
            per = in.op == OP_GATEUP ? g.rt / 2 : g.rt;
        }
        for (int j = 0; j < nt; ++j, ++t) {
            int fail = 0;
            if (lane == 0) {
                if (t >= kPages && !mbar_try_wait(&cx.empty[pg], (use - 1) & 1)) {
                    // the ring is full: use the wait to pull the next tiles into L2
                    while (lc.i < qe && lc.t < t) l2_advance(p, lc, qe);
                    while (lc.i < qe && lc.t < t + la && !mbar_try_wait(&cx.empty[pg], (use - 1) & 1)) {
                        l2_prefetch_tile(p, lc);
                        l2_advance(p, lc, qe);
                    }
                    if (!wait_bar(p, &cx.empty[pg], (use - 1) & 1)) fail = 1;
                }
                // at most `b` tiles in flight (fewer while the consumers poll for
                // an input, so that their loads do not queue behind tile data)
                const uint32_t b = cx.misc->polling ? pback : back;
                if (!fail && t >= b) {
                    const uint32_t tb = t - b;
                    if (!wait_bar(p, &cx.full[tb % kPages], (tb / kPages) & 1)) fail = 1;
                }
                if (fail) cx.misc->aborted = 1;
            }
            if (__shfl_sync(0xFFFFFFFFu, fail, 0)) return;
            uint8_t *dst = cx.pages + (size_t)pg * kPageBytes;
            if (batched && nkc > 1) {
                // one copy per row: the rows' segments [kc*KC, (kc+1)*KC) of a
                // K-chunked tile (gate/up: gate rows, then the up rows from
                // bper rows into the page)
                const BTile bt = batch_tile(j, nrb, nkc, gsz);
                int rows = in.a1 - bt.rb * bper;
                rows = rows < bper ? rows : bper;
                const uint32_t rbytes = (uint32_t)KC * 2;
                const size_t rowlen = (size_t)KC * nkc, coff = (size_t)bt.kc * KC;
                const int halves = in.op == OP_GATEUP ? 2 : 1;
                const size_t row0 = (size_t)in.a0 + (size_t)bt.rb * bper;
                // rows before a matrix boundary of the stacked QKV (the rest
                // come from the next matrix)
                int m = rows;
                if (in.op == OP_QKV) {
                    const size_t qd = (size_t)p.Hq * p.hd, kvd = (size_t)p.Hkv * p.hd;
                    const size_t bound = row0 < qd ? qd : (row0 < qd + kvd ? qd + kvd : qd + 2 * kvd);
                    if (row0 + (size_t)rows > bound) m = (int)(bound - row0);
                }
                bool ok = rows > 0 && CHKS(dst, (uint32_t)(bper * (halves - 1) + rows) * rbytes, 40);
                // sources of the first row of each segment: (half 0 | 1) x (before | after the boundary)
                const uint16_t *s00 = batch_row(p, in, row0, false) + coff;
                const uint16_t *s01 = m < rows ? batch_row(p, in, row0 + m, false) + coff : s00;
                const uint16_t *s10 = halves > 1 ? batch_row(p, in, row0, true) + coff : s00;
                const uint16_t *s11 = s10;
                ok = ok && CHK(s00, rbytes, 3) && CHK(s00 + (size_t)(m - 1) * rowlen, rbytes, 3) &&
                     (m == rows || (CHK(s01, rbytes, 3) && CHK(s01 + (size_t)(rows - m - 1) * rowlen, rbytes, 3))) &&
                     (halves == 1 || (CHK(s10, rbytes, 3) && CHK(s10 + (size_t)(rows - 1) * rowlen, rbytes, 3)));
                if (lane == 0) mbar_expect_tx(&cx.full[pg], ok ? (uint32_t)(halves * rows) * rbytes : 0u);
                __syncwarp();  // the barrier expects the bytes before any copy lands
                if (ok)
                    for (int idx = lane; idx < halves * rows; idx += 32) {
                        const int hf = idx / rows, r = idx % rows;
                        const uint16_t *src = r < m ? (hf ? s10 : s00) + (size_t)r * rowlen
                                                    : (hf ? s11 : s01) + (size_t)(r - m) * rowlen;
                        bulk_g2s(dst + (size_t)(hf * bper + r) * rbytes, src, rbytes, &cx.full[pg], pol);
                    }
                if (lane == 0) cx.misc->n_issued = t + 1;
                if (++pg == kPages) {
                    pg = 0;
                    ++use;
                }
                continue;
            }
            TileCopy c;
            if (batched) {
                c = tile_copy(p, in, batch_tile(j, nrb, 1, gsz).rb);  // one K-chunk: whole rows
            } else if (strided) {
                const size_t off = (size_t)j * per * row_bytes;
                const int rows = in.a1 - j * per < per ? in.a1 - j * per : per;
                c.src0 = static_cast<const uint8_t *>(c0.src0) + off;
                c.src1 = c0.bytes1 ? static_cast<const uint8_t *>(c0.src1) + off : nullptr;
                c.bytes0 = (uint32_t)(rows * row_bytes);
                c.bytes1 = c0.bytes1 ? c.bytes0 : 0u;
                c.dst1 = c0.dst1;
            } else {
                c = tile_copy(p, in, j);
            }
            const bool ok = CHK(c.src0, c.bytes0, 3) && (!c.bytes1 || CHK(c.src1, c.bytes1, 4)) &&
                            CHKS(dst, c.bytes0, 40) && (!c.bytes1 || CHKS(dst + c.dst1, c.bytes1, 41));
            if (lane == 0) {
                mbar_expect_tx(&cx.full[pg], ok ? c.bytes0 + c.bytes1 : 0u);
                if (ok) {
                    bulk_g2s(dst, c.src0, c.bytes0, &cx.full[pg], pol);
                    if (c.bytes1) bulk_g2s(dst + c.dst1, c.src1, c.bytes1, &cx.full[pg], pol);
                }
                cx.misc->n_issued = t + 1;
            }
            if (++pg == kPages) {
                pg = 0;
                ++use;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// GEMV instructions
// ---------------------------------------------------------------------------

// Stages the thread's pairs of a tagged vector of K elements: pair u is
// elements 512*u + 2*tid, +1 (u < NU, those below K), so the threads of a
// warp read one contiguous 256-byte span per load. Every poll reads all of
// the thread's pairs with the loads in flight together, so the round trip
// that sees the last tag also delivers the data (a one-word poll followed
// by the full read measured 9 us/token slower). Returns false on
// abort/timeout.
template <int NU>
__device__ __forceinline__ bool stage_units(const Params &p, const Ctx &cx, const uint2 *src, int K,
                                            uint32_t tag, float &ss) {
    const int t2 = threadIdx.x * 2;
    int last = -1;
#pragma unroll
    for (int u = 0; u < NU; ++u)
        if (512 * u + t2 < K) last = u;
    if (last < 0) return true;
    if (!CHK(src + t2, 16, 38) || !CHK(src + 512 * last + t2, 16, 38)) return false;
    Spin sp;
    while (true) {
        uint4 v[NU];
#pragma unroll
        for (int u = 0; u < NU; ++u)
            v[u] = u <= last ? ll_ld16(src + 512 * u + t2) : make_uint4(0u, tag, 0u, tag);
        bool ok = true;
#pragma unroll
        for (int u = 0; u < NU; ++u) ok = ok && v[u].y == tag && v[u].w == tag;
        if (ok) {
#pragma unroll
            for (int u = 0; u < NU; ++u) {
                if (u > last) continue;
                const float a = __uint_as_float(v[u].x), b = __uint_as_float(v[u].z);
                float *dst = cx.xbuf + 512 * u + t2;
                if (!CHKS(dst, 8, 47)) return false;
                *reinterpret_cast<float2 *>(dst) = make_float2(a, b);
                ss = fmaf(a, a, fmaf(b, b, ss));
            }
            return true;
        }
        if (!sp.keep_going(p)) return false;
    }
}

// Packs two floats as bf16x2, round to nearest even: lo goes to the low half.
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Dot products of two weight rows with the staged input over the warp's
// K-slice (NX*32 columns) on the tensor cores: mma.sync m16n8k16, bf16 in,
// fp32 accumulate. Per 128-column block, A row m < 8 holds the row's
// 16-byte chunks m (k 0-7) and 8+m (k 8-15) and A row 8+m the same chunks
// of the second row (one ldmatrix.x4 over four contiguous 128-byte spans,
// no bank conflicts); B column n holds the inputs of chunks n and 8+n, so
// the diagonal D[m][m] (D[8+m][m]) is chunk pair m's share of the first
// (second) row's dot product, and accumulating over the blocks sums them.
// The input enters as hi and lo bf16 terms (x = hi + lo to 2^-16
// relative): xb holds, per block, this lane's hi pairs at columns 2*lane
// and 64+2*lane, then its lo pairs. wa / wb: the rows at the warp's
// K-slice. On return ra / rb hold the diagonal elements this lane owns (0
// in the other lanes): their warp sums are the two dot products.
template <int NX>
__device__ __forceinline__ void dot_rows2(const uint4 *wa, const uint4 *wb, const uint32_t (&xb)[NX],
                                          float &ra, float &rb) {
    const int lane = threadIdx.x & 31;
    const uint4 *src = ((lane & 8) ? wb : wa) + ((lane & 16) ? 8 : 0) + (lane & 7);
    const uint32_t s0 = smem_u32(src);
    float d[4][4];
#pragma unroll
    for (int c = 0; c < 4; ++c) d[c][0] = d[c][1] = d[c][2] = d[c][3] = 0.f;
#pragma unroll
    for (int b = 0; b < NX / 4; ++b) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(s0 + 256u * b, a0, a1, a2, a3);
        mma_bf16_16816(d[(b & 1) * 2], a0, a1, a2, a3, xb[4 * b], xb[4 * b + 1]);
        mma_bf16_16816(d[(b & 1) * 2 + 1], a0, a1, a2, a3, xb[4 * b + 2], xb[4 * b + 3]);
    }
    float s[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) s[i] = (d[0][i] + d[1][i]) + (d[2][i] + d[3][i]);
    const int g = lane >> 2, t = lane & 3;
    const bool diag = t == (g >> 1), odd = (g & 1) != 0;
    ra = diag ? (odd ? s[1] : s[0]) : 0.f;
    rb = diag ? (odd ? s[3] : s[2]) : 0.f;
}

// Warp sums of two values at once: after the call lanes 0-15 hold the sum of
// a, lanes 16-31 the sum of b (5 shuffles instead of 10).
__device__ __forceinline__ float warp_sum2(float a, float b) {
    const bool hi = (threadIdx.x & 16) != 0;
    const float send = hi ? a : b;
    float v = (hi ? b : a) + __shfl_xor_sync(0xFFFFFFFFu, send, 16);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Stages an input vector of K elements into xbuf (K <= kMaxStaged with
// gains, K <= kMaxStagedLong without): tagged words polled until they carry
// `tag` (or a bf16 row when src_bf is set), the norm gains copied to shared
// memory in the same round trip. Returns the sum of squares of the whole
// vector (valid in every thread) and false on abort/timeout (uniform across
// the consumer warps).
__device__ bool stage_input(const Params &p, const Ctx &cx, const uint2 *src, const uint16_t *src_bf,
                            uint32_t tag, int K, const uint16_t *gain, float &ss_out) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint16_t *gbuf = reinterpret_cast<uint16_t *>(cx.xbuf + kMaxStaged);
    bool ok = src != nullptr || src_bf != nullptr;
    if (tid == 0 && src) cx.misc->polling = 1;
    float ss = 0.f;
    if (gain) {
        for (int i = tid * 8; i < K; i += kConsumerThreads * 8)
            if (CHK(gain + i, 16, 11) && CHKS(gbuf + i, 16, 53))
                *reinterpret_cast<uint4 *>(gbuf + i) = __ldg(reinterpret_cast<const uint4 *>(gain + i));
    }
    if (src_bf) {
        for (int i = tid * 8; i < K; i += kConsumerThreads * 8) {
            uint4 b = make_uint4(0u, 0u, 0u, 0u);
            if (CHK(src_bf + i, 16, 9)) b = __ldg(reinterpret_cast<const uint4 *>(src_bf + i));
            const float v[8] = {bf_lo(b.x), bf_hi(b.x), bf_lo(b.y), bf_hi(b.y),
                                bf_lo(b.z), bf_hi(b.z), bf_lo(b.w), bf_hi(b.w)};
            if (CHKS(cx.xbuf + i, 32, 47)) {
                *reinterpret_cast<float4 *>(cx.xbuf + i) = make_float4(v[0], v[1], v[2], v[3]);
                *reinterpret_cast<float4 *>(cx.xbuf + i + 4) = make_float4(v[4], v[5], v[6], v[7]);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) ss = fmaf(v[e], v[e], ss);
        }
    } else if (ok) {
        // pairs of 512-element units (K <= 8192)
        const int nu = (K + 511) / 512;
        if (nu <= 1) ok = stage_units<1>(p, cx, src, K, tag, ss);
        else if (nu <= 2) ok = stage_units<2>(p, cx, src, K, tag, ss);
        else if (nu <= 4) ok = stage_units<4>(p, cx, src, K, tag, ss);
        else if (nu <= 8) ok = stage_units<8>(p, cx, src, K, tag, ss);
        else ok = stage_units<16>(p, cx, src, K, tag, ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) cx.misc->red8[warp] = ss;
    ok = !consumer_sync_any(!ok);
    if (tid == 0) cx.misc->polling = 0;
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) tot += cx.misc->red8[w];
    ss_out = tot;
    return ok;
}

// One GEMV instruction: rows [a0, a0+a1) of its matrix times the input
// vector, with the op's prologue (RMSNorm) and epilogue (residual,
// SiLU-gate, logits + block argmax). Per-row partial dot products go to
// red[out_index * sw + ks].
template <int NX>
__device__ void gemv_instr(const Params &p, const Ctx &cx, const Instr &in, const Geo &g,
                           uint32_t &t, bool &bad) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rg = warp / g.sw, ks = warp % g.sw;
    const int l = in.layer, n = in.a1, r0 = in.a0;
    const LayerW *lw = p.layers + l;
    const bool gu = in.op == OP_GATEUP;
    const uint32_t ep8 = cx.misc->ep8;
    const uint2 *src = nullptr;
    const uint16_t *src_bf = nullptr, *gain = nullptr;
    uint32_t tag = ep8;
    switch (in.op) {
        case OP_QKV:
            gain = lw->attn_norm;
            if (l == 0)
                src_bf = p.embed + (size_t)current_token(p) * p.d;
            else {
                src = p.xll;
                tag = ep8 | (uint32_t)(2 * l);
            }
            break;
        case OP_GATEUP: gain = lw->mlp_norm; src = p.xll; tag = ep8 | (uint32_t)(2 * l + 1); break;
        case OP_LMHEAD: gain = p.final_norm; src = p.xll; tag = ep8 | (uint32_t)(2 * p.L); break;
        case OP_OPROJ: src = p.attll + (size_t)l * p.Hq * p.hd; break;
        default: src = p.hll + (size_t)l * p.F; break;  // OP_DOWN
    }
    // residual rows of this instruction (O-projection and down; at most one
    // per thread): the load is issued now and checked after the input is
    // staged, so its round trip overlaps the input poll
    const bool has_resid = in.op == OP_OPROJ || in.op == OP_DOWN;
    const uint32_t rtag = ep8 | (uint32_t)(in.op == OP_OPROJ ? 2 * l : 2 * l + 1);
    const bool resid_x = has_resid && !(in.op == OP_OPROJ && l == 0) && tid < n &&
                         CHK(p.xll + r0 + tid, 8, 13);
    uint2 rword = make_uint2(0u, 0u);
    if (resid_x) rword = ll_ld8(p.xll + r0 + tid);
    // this lane's input slice as hi / lo bf16 pairs (see dot_rows2)
    uint32_t xb[NX];
    float *red = in.op == OP_DOWN ? cx.dred : cx.red;
    const int sbase = ks * g.kslice;
    {
        // consecutive instructions of the same op and layer share their input
        const int32_t key = (in.op << 16) | l;
        const bool reuse = cx.misc->staged_key == key;
        float ss = cx.misc->staged_ss;
        if (!reuse && !stage_input(p, cx, bad ? nullptr : src, src_bf, tag, g.K, gain, ss)) bad = true;
        if (has_resid) {
            const int tok = (in.op == OP_OPROJ && l == 0) ? current_token(p) : 0;
            for (int i = tid; i < n; i += kConsumerThreads) {
                float v = 0.f;
                if (in.op == OP_OPROJ && l == 0) {
                    if (CHK(p.embed + (size_t)tok * p.d + r0 + i, 2, 13))
                        v = bf16f(__ldg(p.embed + (size_t)tok * p.d + r0 + i));
                } else if (i == tid && resid_x && rword.y == rtag) {
                    v = __uint_as_float(rword.x);
                } else if (!bad && !ll_read1(p, p.xll + r0 + i, rtag, v)) {
                    bad = true;
                }
                if (CHKS(cx.resid + i, 4, 54)) cx.resid[i] = v;
            }
        }
        bad = consumer_sync_any(bad);
        if (tid == 0) {
            cx.misc->staged_key = bad ? -1 : key;
            cx.misc->staged_ss = ss;
        }
        const float rstd = gain ? 1.0f / sqrtf(ss / (float)g.K + p.eps) : 1.0f;
        const uint16_t *gbuf = reinterpret_cast<const uint16_t *>(cx.xbuf + kMaxStaged);
#pragma unroll
        for (int b = 0; b < NX / 4; ++b)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int idx = sbase + 128 * b + 64 * h + 2 * lane;
                float2 v = *reinterpret_cast<const float2 *>(cx.xbuf + idx);
                if (gain) {
                    const uint32_t gb = *reinterpret_cast<const uint32_t *>(gbuf + idx);
                    v.x *= rstd * bf_lo(gb);
                    v.y *= rstd * bf_hi(gb);
                }
                const uint32_t hi = pack_bf2(v.x, v.y);
                xb[4 * b + h] = hi;
                xb[4 * b + 2 + h] = pack_bf2(v.x - bf_lo(hi), v.y - bf_hi(hi));
            }
    }
    phase_stamp(p, cx, 0);
    // Tiles. Warp (rg, ks) owns rows rg*M .. rg*M+M-1 of every tile (M = 64/NX
    // for every geometry the host plans) and K-slice ks. Everything the loop
    // needs is copied into registers first: values read through `p` or `g`
    // live in shared memory and would be reloaded after every barrier op.
    constexpr int M = 64 / NX;
    const int sw = g.sw;
    const int per = gu ? g.rt / 2 : g.rt;
    const int nt = (n + per - 1) / per;
    const int row_u4 = g.K / 8;  // 16-byte chunks per row
    const bool tracing = p.trace != nullptr;
    const uint4 *pages = reinterpret_cast<const uint4 *>(cx.pages);
    const int woff = rg * M * row_u4 + sbase / 8;  // the warp's first row at its K-slice
    const bool second = (lane & 16) != 0;  // lanes 16-31 hold the second row's sum
    // row r of a tile is output row j*per + roff[r] (+ n for the up half of a gate/up tile)
    int roff[M], obase[M];
#pragma unroll
    for (int q = 0; q < M; ++q) {
        const int r = rg * M + q;
        const bool up = gu && r >= per;
        roff[q] = up ? r - per : r;
        obase[q] = up ? n : 0;
    }
    int pg = (int)(t % kPages);
    uint32_t par = (t / kPages) & 1u;
    for (int j = 0; j < nt; ++j) {
        if (!bad && !wait_tile(p, cx, pg, par, tracing)) bad = true;
        bad = __any_sync(0xFFFFFFFFu, bad);  // warp-uniform from here on
        bool released = false;
        if (!bad) {
            const uint4 *page = pages + pg * (kPageBytes / 16) + woff;
#pragma unroll
            for (int q = 0; q < M; q += 2) {
                const int row0 = j * per + roff[q], row1 = j * per + roff[q + 1];
                const bool v0 = row0 < n, v1 = row1 < n;
                if (!v0 && !v1) continue;
                const uint4 *wa = page + q * row_u4;
                const uint4 *wb = v1 ? wa + row_u4 : wa;  // an invalid second row re-reads the first
                float ra = 0.f, rb = 0.f;
                if (CHKS(wa, 16, 44) && CHKS(wa + 4 * NX - 1, 16, 45) && CHKS(wb, 16, 44) &&
                    CHKS(wb + 4 * NX - 1, 16, 45))
                    dot_rows2<NX>(wa, wb, xb, ra, rb);
                // with one row pair per warp the page is free once the weights are in registers
                if (M == 2) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&cx.empty[pg]);
                    released = true;
                }
                const float sum = warp_sum2(ra, rb);
                const bool vh = second ? v1 : v0;
                const int oh = second ? obase[q + 1] + row1 : obase[q] + row0;
                if ((lane & 15) == 0 && vh && CHKS(red + oh * sw + ks, 4, 46)) red[oh * sw + ks] = sum;
            }
        }
        if (!released) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&cx.empty[pg]);
        }
        ++t;
        if (++pg == kPages) {
            pg = 0;
            par ^= 1u;
        }
    }
}

// ---------------------------------------------------------------------------
// Filtered draw (top-k / top-p) in the LM-head epilogue.
// ---------------------------------------------------------------------------
// The logit and the vocabulary index held in an argmax key.
__device__ __forceinline__ float key_value(unsigned long long k) {
    uint32_t u = (uint32_t)(k >> 32);
    u = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
    return __uint_as_float(u);
}
__device__ __forceinline__ uint32_t key_index(unsigned long long k) { return 0xFFFFFFFFu - (uint32_t)k; }

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        v = w > v ? w : v;
    }
    return v;
}

// 64 keys held by a warp, element e = lane + 32 r in v[r]: one compare-exchange
// stage of a bitonic network over distance j within blocks of size k
// (descending overall: blocks with (e & k) == 0 descend).
__device__ __forceinline__ void bitonic_stage64(unsigned long long (&v)[2], int k, int j) {
    const int lane = threadIdx.x & 31;
    if (j == 32) {  // the partner is the lane's other element
        const bool desc = (lane & k) == 0;  // e = lane and lane + 32 share the block bit for k >= 64
        const unsigned long long hi = v[0] > v[1] ? v[0] : v[1], lo = v[0] > v[1] ? v[1] : v[0];
        v[0] = desc ? hi : lo;
        v[1] = desc ? lo : hi;
        return;
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int e = lane + 32 * r;
        const unsigned long long pv = __shfl_xor_sync(0xFFFFFFFFu, v[r], j);
        const bool desc = (e & k) == 0, lower = (e & j) == 0;
        const unsigned long long mx = v[r] > pv ? v[r] : pv, mn = v[r] > pv ? pv : v[r];
        v[r] = lower == desc ? mx : mn;
    }
}

// Sorts the warp's 64 keys descending.
__device__ __forceinline__ void warp_sort64(unsigned long long (&v)[2]) {
#pragma unroll
    for (int k = 2; k <= 64; k <<= 1)
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) bitonic_stage64(v, k, j);
}

// Two descending runs of 64 (a, then b) -> the 64 largest keys of both,
// descending, in a: the elementwise max of a and reversed b is bitonic and
// holds them, and a bitonic merge sorts it.
__device__ __forceinline__ void warp_merge_top64(unsigned long long (&a)[2], const unsigned long long (&b)[2]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const unsigned long long rb = __shfl_sync(0xFFFFFFFFu, b[1 - r], 31 - lane);  // b[63 - e]
        a[r] = a[r] > rb ? a[r] : rb;
    }
#pragma unroll
    for (int j = 32; j > 0; j >>= 1) bitonic_stage64(a, 64, j);
}

// The 64 largest of keys[0 .. n), descending, into keys[0 .. 64) (0 pads
// the rest; no real key is 0), by the consumer warps: each warp sorts runs of
// 64 in registers and keeps the best 64 of its two runs, then rounds of
// pairwise keep-the-best-64 merges leave the survivors in run 0. keys must
// hold max(n, 64) entries. Ends with the consumers synchronised.
__device__ void block_top64(unsigned long long *keys, int n) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nrun = n > 64 ? (n + 63) / 64 : 1;
    const int cap = n > 64 ? n : 64;  // entries that may be written (a short last run keeps its real keys)
    unsigned long long v[2], w2[2];
    auto load_run = [&](int run, unsigned long long (&x)[2]) {
        const int base = run * 64;
        x[0] = base + lane < n ? keys[base + lane] : 0ull;
        x[1] = base + lane + 32 < n ? keys[base + lane + 32] : 0ull;
    };
    for (int pair = warp; 2 * pair < nrun; pair += kConsumerWarps) {
        load_run(2 * pair, v);
        warp_sort64(v);
        if (2 * pair + 1 < nrun) {
            load_run(2 * pair + 1, w2);
            warp_sort64(w2);
            warp_merge_top64(v, w2);
        }
        __syncwarp();
        if (2 * pair * 64 + lane < cap) keys[2 * pair * 64 + lane] = v[0];
        if (2 * pair * 64 + lane + 32 < cap) keys[2 * pair * 64 + lane + 32] = v[1];
    }
    consumer_sync();
    for (int step = 2; step < nrun; step <<= 1) {  // runs 0, 2 step, 4 step, ... hold the survivors
        for (int pair = warp; 2 * pair * step < nrun; pair += kConsumerWarps) {
            const int r0 = 2 * pair * step, r1 = r0 + step;
            if (r1 < nrun) {  // r0 < r1: never the short last run, so 64 entries fit
                load_run(r0, v);
                load_run(r1, w2);
                warp_merge_top64(v, w2);
                __syncwarp();
                keys[r0 * 64 + lane] = v[0];
                keys[r0 * 64 + lane + 32] = v[1];
            }
        }
        consumer_sync();
    }
}

// The filtered draw from nl candidate lists (list s at lists + s * kMaxTopK:
// the top_k best keys of its part of the vocabulary in descending order, 0
// where it has fewer), by the consumer threads of one CTA. tau = the top_k-th
// largest of the lists' J = ceil(top_k / nl) best keys is a lower bound of
// the global top_k (those keys are some of the candidates); every key >= tau
// (a prefix of each list) is gathered into g, their top_k selected, and warp 0
// cuts the nucleus (the shortest prefix of the top_k whose softmax mass at
// the temperature reaches top_p) and takes the Gumbel-max among the kept
// candidates with the noise of (entry, pos, slot, seed). g: shared memory for
// max(nl * top_k, 64) keys; gcount: a shared int. Returns the token in warp 0
// (-1 in the other warps).
__device__ int draw_filtered(const unsigned long long *lists, int nl, int K, float top_p, float inv_temp, int pos,
                             int slot, uint32_t seed_lo, uint32_t seed_hi, unsigned long long *g, int *gcount) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned long long tau = 0ull;
    {
        const int J = (K + nl - 1) / nl, ns = nl * J;
        if (tid == 0) *gcount = 0;
        for (int e = tid; e < ns; e += kConsumerThreads) g[e] = __ldcg(lists + (size_t)(e / J) * kMaxTopK + e % J);
        consumer_sync();
        block_top64(g, ns);
        tau = K - 1 < ns ? g[K - 1] : 0ull;
        consumer_sync();  // g is reused below
    }
    // every list's prefix of keys >= tau (a thread per list)
    for (int s = tid; s < nl; s += kConsumerThreads) {
        const unsigned long long *q = lists + (size_t)s * kMaxTopK;
        for (int j = 0; j < K; ++j) {
            const unsigned long long v = __ldcg(q + j);
            if (v == 0ull || v < tau) break;
            g[atomicAdd(gcount, 1)] = v;
        }
    }
    consumer_sync();
    const int ng = *(volatile int *)gcount;
    block_top64(g, ng);  // the top k of the candidates, descending, in g[0 .. k)
    if (warp != 0) return -1;
    // warp 0: candidate j = lane and j = lane + 32 (K <= 64), in key order
    const int nc = ng < K ? ng : K;
    const float zmax = key_value(g[0]);
    const bool h0 = lane < nc, h1 = lane + 32 < nc;
    const float z0 = h0 ? key_value(g[lane]) : 0.f, z1 = h1 ? key_value(g[lane + 32]) : 0.f;
    const float e0 = h0 ? expf((z0 - zmax) * inv_temp) : 0.f, e1 = h1 ? expf((z1 - zmax) * inv_temp) : 0.f;
    float c0 = e0, c1 = e1;  // inclusive prefix sums in candidate order
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float a = __shfl_up_sync(0xFFFFFFFFu, c0, o), b = __shfl_up_sync(0xFFFFFFFFu, c1, o);
        if (lane >= o) {
            c0 += a;
            c1 += b;
        }
    }
    c1 += __shfl_sync(0xFFFFFFFFu, c0, 31);
    const float need = top_p * __shfl_sync(0xFFFFFFFFu, c1, 31);
    int nkeep = nc;
    if (top_p < 1.f) {
        const uint32_t b0 = __ballot_sync(0xFFFFFFFFu, h0 && c0 >= need);
        const uint32_t b1 = __ballot_sync(0xFFFFFFFFu, h1 && c1 >= need);
        nkeep = b0 ? __ffs(b0) : (b1 ? 32 + __ffs(b1) : nc);
    }
    unsigned long long best = 0ull;
    if (lane < nkeep) {
        const uint32_t i = key_index(g[lane]);
        best = argmax_key(z0 * inv_temp + gumbel_noise(i, pos, slot, seed_lo, seed_hi), i);
    }
    if (lane + 32 < nkeep) {
        const uint32_t i = key_index(g[lane + 32]);
        const unsigned long long k1 = argmax_key(z1 * inv_temp + gumbel_noise(i, pos, slot, seed_lo, seed_hi), i);
        best = k1 > best ? k1 : best;
    }
    best = warp_max_u64(best);
    return (int)key_index(best);
}

// LM-head epilogue of a filtered draw. Every LM-head instruction selects the
// top_k best keys (logit, then lowest index) of its rows, in order, and
// publishes them; the last instruction to arrive bounds the global top_k from
// below by the top_k-th largest of the blocks' best keys, gathers the
// published keys at or above that bound, selects their top_k, and with warp 0
// cuts the nucleus (the shortest prefix of the top_k whose softmax mass at
// the temperature reaches top_p) and takes the Gumbel-max among the kept
// candidates.
__device__ void lm_filtered(const Params &p, const Ctx &cx, const Instr &in, const float *red, int sw) {
    const int tid = threadIdx.x;
    const int n = in.a1, r0 = in.a0, K = p.top_k;
    unsigned long long *keys = reinterpret_cast<unsigned long long *>(cx.xbuf);  // n <= 1024 keys (8 KB)
    if (tid == 0) cx.misc->staged_key = -1;  // xbuf stops holding the staged input
    int np = 2;
    while (np < n || np < K) np <<= 1;
    for (int i = tid; i < np; i += kConsumerThreads) {
        unsigned long long k = 0ull;  // no real key is 0
        if (i < n) {
            float v = 0.f;
            for (int s = 0; s < sw; ++s) v += red[i * sw + s];
            if (p.out_logits && CHK(p.out_logits + r0 + i, 4, 18)) p.out_logits[r0 + i] = v;
            k = argmax_key(v, (uint32_t)(r0 + i));
        }
        if (CHKS(keys + i, 8, 62)) keys[i] = k;
    }
    consumer_sync();
    block_top64(keys, np);
    unsigned long long *mine = p.lm_cand + (size_t)in.slot * kMaxTopK;
    for (int j = tid; j < K; j += kConsumerThreads)
        if (CHK(mine + j, 8, 63)) mine[j] = keys[j];
    consumer_sync();
    if (tid == 0) {
        __threadfence();
        const uint32_t old = CHK(p.ctr + p.cl.lm_arrive, 4, 31) ? atom_acq_rel_add(p.ctr + p.cl.lm_arrive, 1u) : 0u;
        const bool last = old == (uint32_t)p.n_lm - 1u;
        if (last) __threadfence();
        cx.misc->flag = last ? 1 : 0;
        cx.misc->gcount = 0;
    }
    consumer_sync();
    if (!cx.misc->flag) return;
    const int tok = draw_filtered(p.lm_cand, p.n_lm, K, p.top_p, p.inv_temp, p.pos, p.bslot, p.seed_lo, p.seed_hi,
                                  reinterpret_cast<unsigned long long *>(cx.pages), &cx.misc->gcount);
    if (tid == 0 && CHK(p.out_token, 4, 21)) *p.out_token = tok;
}

__device__ void do_gemv(const Params &p, const Ctx &cx, const Instr &in, uint32_t &t, bool &bad) {
    const Geo &g = geo_of(p, in.op);
    const int tid = threadIdx.x;
    const int l = in.layer;
    switch (g.nx) {  // the host plans every operand with nx in {8, 16, 24, 32}
        case 8: gemv_instr<8>(p, cx, in, g, t, bad); break;
        case 16: gemv_instr<16>(p, cx, in, g, t, bad); break;
        case 24: gemv_instr<24>(p, cx, in, g, t, bad); break;
        default: gemv_instr<32>(p, cx, in, g, t, bad); break;
    }
    phase_stamp(p, cx, 1);
    bad = consumer_sync_any(bad);
    if (bad) return;
    // ---- epilogue: combine K-slices, apply the op's output transform
    const int n = in.a1, r0 = in.a0, sw = g.sw;
    const uint32_t ep8 = cx.misc->ep8;
    const float *red = in.op == OP_DOWN ? cx.dred : cx.red;
    switch (in.op) {
        case OP_QKV: {
            uint2 *dst = p.qkvll + (size_t)l * (p.Hq + 2 * p.Hkv) * p.hd + r0;  // stacked q | k | v
            for (int i = tid; i < n; i += kConsumerThreads) {
                float v = 0.f;
                for (int s = 0; s < sw; ++s) v += red[i * sw + s];
                if (CHK(dst + i, 8, 12)) ll_store(dst + i, v, ep8);
            }
            break;
        }
        case OP_OPROJ:
        case OP_DOWN: {
            const uint32_t wtag = ep8 | (uint32_t)(in.op == OP_OPROJ ? 2 * l + 1 : 2 * l + 2);
            for (int i = tid; i < n; i += kConsumerThreads) {
                float v = 0.f;
                for (int s = 0; s < sw; ++s) v += red[i * sw + s];
                if (CHK(p.xll + r0 + i, 8, 15)) ll_store(p.xll + r0 + i, cx.resid[i] + v, wtag);
            }
            break;
        }
        case OP_GATEUP: {
            uint2 *dst = p.hll + (size_t)l * p.F + r0;
            for (int i = tid; i < n; i += kConsumerThreads) {
                float gv = 0.f, uv = 0.f;
                for (int s = 0; s < sw; ++s) {
                    gv += red[i * sw + s];
                    uv += red[(n + i) * sw + s];
                }
                if (CHK(dst + i, 8, 16)) ll_store(dst + i, gv / (1.0f + expf(-gv)) * uv, ep8);
            }
            break;
        }
        default: {  // OP_LMHEAD
            if (p.top_k > 0 && p.inv_temp > 0.f) {
                lm_filtered(p, cx, in, red, sw);
                break;
            }
            unsigned long long best = 0ull;
            for (int i = tid; i < n; i += kConsumerThreads) {
                float v = 0.f;
                for (int s = 0; s < sw; ++s) v += red[i * sw + s];
                if (p.out_logits && CHK(p.out_logits + r0 + i, 4, 18)) p.out_logits[r0 + i] = v;
                const float z = p.inv_temp > 0.f
                                    ? v * p.inv_temp + gumbel_noise((uint32_t)(r0 + i), p.pos, p.bslot, p.seed_lo, p.seed_hi)
                                    : v;
                const unsigned long long k = argmax_key(z, (uint32_t)(r0 + i));
                best = k > best ? k : best;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, best, o);
                best = other > best ? other : best;
            }
            const int warp = tid >> 5;
            if ((tid & 31) == 0) cx.misc->best8[warp] = best;
            consumer_sync();
            if (tid == 0) {
                unsigned long long b = 0ull;
                for (int w = 0; w < kConsumerWarps; ++w) b = cx.misc->best8[w] > b ? cx.misc->best8[w] : b;
                if (CHK(p.lm_part + in.slot, 8, 19)) p.lm_part[in.slot] = b;
                // the last LM-head instruction to arrive reduces all block maxima
                const uint32_t old = CHK(p.ctr + p.cl.lm_arrive, 4, 31)
                                         ? atom_acq_rel_add(p.ctr + p.cl.lm_arrive, 1u) : 0u;
                const bool last = old == (uint32_t)p.n_lm - 1u;
                if (last) __threadfence();
                cx.misc->flag = last ? 1 : 0;
            }
            consumer_sync();
            if (cx.misc->flag) {
                // all consumer threads load the block maxima at once
                unsigned long long g2 = 0ull;
                for (int s = tid; s < p.n_lm; s += kConsumerThreads) {
                    const unsigned long long v = CHK(p.lm_part + s, 8, 20) ? __ldcg(p.lm_part + s) : 0ull;
                    g2 = v > g2 ? v : g2;
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, g2, o);
                    g2 = other > g2 ? other : g2;
                }
                if ((tid & 31) == 0) cx.misc->best8[warp] = g2;
                consumer_sync();
                if (tid == 0) {
                    unsigned long long b = 0ull;
                    for (int w = 0; w < kConsumerWarps; ++w) b = cx.misc->best8[w] > b ? cx.misc->best8[w] : b;
                    if (CHK(p.out_token, 4, 21))
                        *p.out_token = (int32_t)(0xFFFFFFFFu - (uint32_t)(b & 0xFFFFFFFFull));
                }
            }
            break;
        }
    }
}

// ---------------------------------------------------------------------------
// Batched GEMV (nb > 1 sequences in one step, every weight read once): a
// real contraction Y[rows, nb] = W X^T, on the tensor cores with mma.sync
// m16n8k16 (fp16 in, fp32 accumulate): A = 16 weight rows from the handle's
// fp16 copy of the bf16 weights (exact in fp16's normal range), B = the 8
// sequences' inputs rounded to fp16 (relative error <= 2^-11), D in
// registers.
// Tile = rt rows x a K-chunk of KC = g.pad columns (32 KB). Warp (rg, ks)
// owns 16 rows of every tile (the MMA's A rows; for gate/up 8 gate rows and
// the matching 8 up rows) and the 128-wide slice ks of the chunk: 8 MMAs per
// tile, its inputs in 16 registers. The k order inside each
// 32-column block is permuted identically for X and W so that every lane
// reads 16 contiguous bytes of a weight row. Lanes add their (sequence, row)
// sums into a shared accumulator; the last warp to finish a tile of the last
// K-chunk (an arrival counter per tile) applies the op's transform and
// publishes the tile's outputs, with no CTA-wide barrier per tile. The
// RMSNorm factor of a sequence is a scalar of the whole row, so it is
// applied there too, from the sums of squares the warps gathered while
// loading their slices.
// Tile order: K-chunk by K-chunk over all row blocks when the instruction's
// accumulators fit in shared memory; otherwise (more rows per instruction
// than the accumulators hold) groups of 8 row
// blocks, all K-chunks of a group before the next, through a ring of 8
// accumulator slots (a warp runs at most kPages tiles ahead of the slowest,
// and a slot is reused 8 tiles later).
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t f2h(float f) { return (uint32_t)__half_as_ushort(__float2half_rn(f)); }

// Reads elements e0 + 32*c + j (c = 0..3, j = 0..7) of one sequence from an
// interleaved batched buffer, e0 = 8t: q = buffer + bofs(b, e0), the four
// elements from 32*c + 4*h at q + 256*c + 128*h. All 8 loads go out together.
__device__ __forceinline__ void ld_blocks4(const float *q, float (&out)[4][8]) {
    float4 v[4][2];
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int h = 0; h < 2; ++h) v[c][h] = ld_relaxed_f4(q + 256 * c + 128 * h);
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            out[c][4 * h] = v[c][h].x;
            out[c][4 * h + 1] = v[c][h].y;
            out[c][4 * h + 2] = v[c][h].z;
            out[c][4 * h + 3] = v[c][h].w;
        }
}

// Completion counters of the batched steps: an instruction that waits on
// one spins (thread 0, acquire) until it reaches its target, then the
// consumers' barrier orders everyone's reads after it; a producing
// instruction releases its counters after a barrier over its writers.
__device__ __forceinline__ bool ctr_wait(const Params &p, int idx, uint32_t target) {
    if (idx < 0 || !CHK(p.ctr + idx, 4, 60)) return true;
    Spin sp;
    while (ld_acquire(p.ctr + idx) < target)
        if (!sp.keep_going(p)) return false;
    return true;
}

__device__ __forceinline__ void ctr_signal(const Params &p, int idx, int n) {
    __threadfence();
    for (int k = 0; k < n; ++k)
        if (CHK(p.ctr + idx + k, 4, 61)) red_release_add(p.ctr + idx + k, 1u);
}

__device__ bool gemv_batch(const Params &p, const Ctx &cx, const Instr &in, uint32_t &t, bool &bad) {
    const Geo &g = geo_of(p, in.op);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int sw = g.sw, rg = warp / sw, ks = warp % sw;
    const int K = g.K, KC = g.pad, nkc = K / KC, R = g.rt;
    const int l = in.layer, n = in.a1, r0 = in.a0, op = in.op, nb = p.nb;
    const bool gu = op == OP_GATEUP;
    const int per = gu ? R / 2 : R;  // output rows per tile
    const int nrb = (n + per - 1) / per;
    const bool ring = batch_ring(n, op);
    const int gsz = ring ? 8 : nrb;
    const int nt = nrb * nkc;
    const uint32_t ep8 = cx.misc->ep8;
    const LayerW *lw = p.layers + l;
    const int gq = lane >> 2, tq = lane & 3;  // MMA fragment coordinates
    // inputs: interleaved fp32 buffers (bofs), or the bf16 embedding rows (layer-0 QKV)
    float *const xf = reinterpret_cast<float *>(p.xll);
    float *const hf = reinterpret_cast<float *>(p.hll) + (size_t)l * kMaxBatch * p.F;
    const float *src = nullptr;
    const uint16_t *gain = nullptr;
    const bool emb = op == OP_QKV && l == 0;
    switch (op) {
        case OP_QKV: gain = lw->attn_norm; src = xf; break;
        case OP_GATEUP: gain = lw->mlp_norm; src = xf; break;
        case OP_OPROJ: src = reinterpret_cast<const float *>(p.attll) + (size_t)l * kMaxBatch * p.Hq * p.hd; break;
        default: src = hf; break;  // OP_DOWN
    }
    float *acc = cx.xbuf;                          // kBatchAcc floats: xbuf and red
    int *cnt = reinterpret_cast<int *>(cx.dred);  // ring: arrivals per slot
    float *resid = cx.resid;                       // [nb][n] residual rows (O-proj, down)
    float *ssum = cx.misc->red8;                   // [kMaxBatch] sums of squares of the inputs
    {
        const int na = ring ? 8 * R * kMaxBatch : n * (gu ? 2 : 1) * kMaxBatch;
        for (int i = tid; i < na; i += kConsumerThreads)
            if (CHKS(acc + i, 4, 55)) acc[i] = 0.f;
        if (ring && tid < 8 && CHKS(cnt + tid, 4, 56)) cnt[tid] = 0;
        if (tid < kMaxBatch) ssum[tid] = 0.f;
    }
    // this instruction's inputs are complete once its wait counter is
    if (tid == 0 && !bad && !ctr_wait(p, in.wait_ctr, (uint32_t)in.wait_target)) bad = true;
    bad = consumer_sync_any(bad);
    if (bad) return true;
    if (op == OP_OPROJ || op == OP_DOWN) {  // residual rows of every sequence
        for (int i = tid; i < n * nb; i += kConsumerThreads) {
            const int b = i / n, r = i % n;
            float v;
            if (op == OP_OPROJ && l == 0) {
                const int tok = current_token(p, b);
                v = CHK(p.embed + (size_t)tok * p.d + r0 + r, 2, 13) ? bf16f(__ldg(p.embed + (size_t)tok * p.d + r0 + r)) : 0.f;
            } else {
                v = CHK(xf + bofs(b, r0 + r), 4, 14) ? ld_relaxed_f(xf + bofs(b, r0 + r)) : 0.f;
            }
            if (CHKS(resid + i, 4, 54)) resid[i] = v;
        }
    }
    // This lane's inputs: sequence gq, elements 32*c + 8*tq .. +8 of the
    // warp's slice (c = 0..3), times the norm gain, as fp16 pairs: the B
    // fragments of all 8 MMAs of a tile. Sequences >= nb are zero.
    uint32_t xb[4][4];
    auto load_inputs = [&](int kc, bool first) -> bool {
        float xv[4][8];
        const int e0 = kc * KC + ks * 128 + 8 * tq;  // + 32 * c
        bool ok = true;
        if (gq >= nb) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int e = 0; e < 8; ++e) xv[c][e] = 0.f;
        } else if (emb) {
            const uint16_t *row = p.embed + (size_t)current_token(p, gq) * p.d + e0;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint4 w = make_uint4(0u, 0u, 0u, 0u);
                if (CHK(row + 32 * c, 16, 9)) w = __ldg(reinterpret_cast<const uint4 *>(row + 32 * c));
                xv[c][0] = bf_lo(w.x); xv[c][1] = bf_hi(w.x); xv[c][2] = bf_lo(w.y); xv[c][3] = bf_hi(w.y);
                xv[c][4] = bf_lo(w.z); xv[c][5] = bf_hi(w.z); xv[c][6] = bf_lo(w.w); xv[c][7] = bf_hi(w.w);
            }
        } else if (CHK(src + bofs(gq, e0), 16, 38) && CHK(src + bofs(gq, e0) + 896, 16, 38)) {
            ld_blocks4(src + bofs(gq, e0), xv);
        } else {
            ok = false;
        }
        if (gain) {
            if (first && rg == 0) {  // each chunk's squares once (row group 0); lanes 4g .. 4g+3 hold sequence g
                float ss = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int e = 0; e < 8; ++e) ss = fmaf(xv[c][e], xv[c][e], ss);
                ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 1);
                ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 2);
                if (tq == 0 && gq < nb) atomicAdd(ssum + gq, ss);
            }
            const uint16_t *gp = gain + e0;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint4 gw = make_uint4(0u, 0u, 0u, 0u);
                if (CHK(gp + 32 * c, 16, 11)) gw = __ldg(reinterpret_cast<const uint4 *>(gp + 32 * c));
                xv[c][0] *= bf_lo(gw.x); xv[c][1] *= bf_hi(gw.x); xv[c][2] *= bf_lo(gw.y); xv[c][3] *= bf_hi(gw.y);
                xv[c][4] *= bf_lo(gw.z); xv[c][5] *= bf_hi(gw.z); xv[c][6] *= bf_lo(gw.w); xv[c][7] *= bf_hi(gw.w);
            }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int k = 0; k < 4; ++k)
                xb[c][k] = f2h(xv[c][2 * k]) | (f2h(xv[c][2 * k + 1]) << 16);
        return ok;
    };
    phase_stamp(p, cx, 0);
    // this warp's 16 rows of a tile: this lane loads the A rows gq (trow0)
    // and gq + 8 (trow1); for gate/up they are the gate row and the up row
    // of the same output
    const int ra0 = gu ? rg * 8 : rg * 16;
    const int trow0 = ra0 + gq, trow1 = gu ? per + ra0 + gq : ra0 + 8 + gq;
    const int row_u4 = KC / 8;
    const uint4 *pages = reinterpret_cast<const uint4 *>(cx.pages);
    const int woff0 = trow0 * row_u4 + ks * 16 + tq, woff1 = trow1 * row_u4 + ks * 16 + tq;  // + 4 * c
    const bool tracing = p.trace != nullptr;
    // Applies the op's transform to output row o (of the instruction) of
    // sequence b, accumulator row arow, and publishes it.
    auto publish = [&](int o, int b, int arow, float rs) {
        const float v = acc[arow * kMaxBatch + b] * rs;
        if (op == OP_QKV) {
            uint2 *dst = p.qkvll + ((size_t)l * nb + b) * (p.Hq + 2 * p.Hkv) * p.hd + r0 + o;
            if (CHK(dst, 8, 12)) ll_store(dst, v, ep8);
        } else if (op == OP_OPROJ || op == OP_DOWN) {
            float *dst = xf + bofs(b, r0 + o);
            if (CHK(dst, 4, 15)) *dst = resid[b * n + o] + v;
        } else {  // gate/up
            const float up = acc[(arow + 1) * kMaxBatch + b] * rs;
            float *dst = hf + bofs(b, r0 + o);
            if (CHK(dst, 4, 16)) *dst = v / (1.0f + expf(-v)) * up;
        }
    };
    int pg = (int)(t % kPages);
    uint32_t par = (t / kPages) & 1u;
    int cur = -1;  // (group, K-chunk) whose inputs the registers hold
    for (int j = 0; j < nt; ++j) {
        const BTile bt = batch_tile(j, nrb, nkc, gsz);
        const int rb = bt.rb, grp = rb / gsz;
        const int key = grp * nkc + bt.kc;
        if (key != cur) {
            if (!bad && !load_inputs(bt.kc, grp == 0)) bad = true;
            cur = key;
        }
        const bool last_chunk = bt.kc == nkc - 1;
        if (!bad && !wait_tile(p, cx, pg, par, tracing)) bad = true;
        bad = __any_sync(0xFFFFFFFFu, bad);
        const int slot = ring ? (rb & 7) : rb;
        if (!bad) {
            const uint4 *page = pages + pg * (kPageBytes / 16);
            uint4 w0[4], w1[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                w0[c] = page[woff0 + 4 * c];
                w1[c] = page[woff1 + 4 * c];
            }
            __syncwarp();  // the page is free once its weights are in registers
            if (lane == 0) mbar_arrive(&cx.empty[pg]);
            // A = 16 weight rows (this lane: rows gq and gq + 8), B = the 8
            // sequences' inputs; D rows gq / gq + 8, columns (sequences) 2tq, 2tq+1
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                mma_f16_16816(d, w0[c].x, w1[c].x, w0[c].y, w1[c].y, xb[c][0], xb[c][1]);
                mma_f16_16816(d, w0[c].z, w1[c].z, w0[c].w, w1[c].w, xb[c][2], xb[c][3]);
            }
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const int blk = h >> 1, b = 2 * tq + (h & 1);  // weight row block (gq / gq + 8), sequence
                int o, arow;  // output row within the tile, accumulator row
                if (gu) {
                    o = ra0 + gq;
                    arow = ((ring ? slot : rb) * per + o) * 2 + blk;
                } else {
                    o = ra0 + 8 * blk + gq;
                    arow = (ring ? slot * R : rb * per) + o;
                }
                if (b < nb && rb * per + o < n && CHKS(acc + arow * kMaxBatch + b, 4, 58))
                    atomicAdd(acc + arow * kMaxBatch + b, d[h]);
            }
        } else {
            __syncwarp();
            if (lane == 0) mbar_arrive(&cx.empty[pg]);
        }
        ++t;
        if (++pg == kPages) {
            pg = 0;
            par ^= 1u;
        }
        if (!ring || !last_chunk) continue;
        // ring: the last warp to finish a tile of the last K-chunk publishes
        // its rows and frees the slot
        __threadfence_block();
        __syncwarp();
        int old = 0;
        if (lane == 0 && CHKS(cnt + slot, 4, 59)) old = atomicAdd(cnt + slot, 1);
        old = __shfl_sync(0xFFFFFFFFu, old, 0);
        if (old != kConsumerWarps - 1 || bad) continue;
        __threadfence_block();
        {
            const int b = lane & 7;  // the sequence of every element this lane publishes
            const float rs = gain && b < nb ? 1.0f / sqrtf(ssum[b] / (float)K + p.eps) : 1.0f;
            for (int idx = lane; idx < per * kMaxBatch; idx += 32) {
                const int i = idx / kMaxBatch;
                const int arow = gu ? (slot * per + i) * 2 : slot * R + i;
                if (b < nb && rb * per + i < n) publish(rb * per + i, b, arow, rs);
                acc[arow * kMaxBatch + b] = 0.f;
                if (gu) acc[(arow + 1) * kMaxBatch + b] = 0.f;
            }
        }
        if (lane == 0) cnt[slot] = 0;
        __threadfence_block();
    }
    if (!ring) {
        // all tiles accumulated: every thread publishes rows of one sequence
        bad = consumer_sync_any(bad);
        if (bad) return true;
        const int b = tid & 7;
        const float rs = gain && b < nb ? 1.0f / sqrtf(ssum[b] / (float)K + p.eps) : 1.0f;
        if (b < nb)
            for (int i = tid >> 3; i < n; i += kConsumerThreads / kMaxBatch) publish(i, b, gu ? 2 * i : i, rs);
    }
    // O-proj, gate/up and down release their completion counters (QKV's
    // outputs are tagged words that the attention waits on)
    if (op == OP_OPROJ || op == OP_GATEUP || op == OP_DOWN) {
        bad = consumer_sync_any(bad);
        if (bad) return true;
        if (tid == 0) ctr_signal(p, in.sig_ctr, in.sig_n);
    }
    phase_stamp(p, cx, 1);
    return false;
}

template <int HD, int G>
struct AttnWarpState {
    // running max (log2 units) and sum of the head this lane scores
    // (head dq % GP of the score layout), the same in every lane of that head
    float m, l;
    // lane (pv, dg) of the P.V layout: unnormalised output dims dg*8..dg*8+7
    // of every head, summed over the positions pv, pv + PGV, ... it saw
    float o[G][8];
};

// Lane layouts of one chunk of up to 32 positions:
//  scores: lane = (position pl, dim group dq): DQ = HD/16 groups of 16 dims,
//          PG = 32/DQ positions per pass, NPASS passes. A lane multiplies its
//          16 dims for all heads, then a reduce-scatter over the dim groups
//          leaves it the full score of head dq % GP (GP = G, or 4 for G = 3).
//  P.V:    lane = (position group pv, dim group dg): DGV = HD/8 groups of 8 dims,
//          PGV = 32/DGV groups; a lane walks positions pv, pv + PGV, ...
template <int HD, int G>
struct AttnLayout {
    static constexpr int DQ = HD / 16, PG = 32 / DQ, NPASS = 32 / PG;
    static constexpr int DGV = HD / 8, PGV = 32 / DGV;
    static constexpr int GP = G == 3 ? 4 : G;
    // q in shared memory: head g, dim d at g*QSTR + (d/16)*20 + d%16; the
    // 4-float pad puts the dim groups read together on different banks
    static constexpr int QSTR = HD / 16 * 20;
    static __device__ __forceinline__ int qidx(int g, int d) { return g * QSTR + (d >> 4) * 20 + (d & 15); }
};

// One chunk of up to 32 positions for this warp. Kp/Vp point at the chunk's
// first key/value row (bf16, HD each); npos valid positions; q holds the G
// pre-scaled query heads (fp32, shared, AttnLayout::qidx); pbuf is this warp's
// [32][4] scratch for the softmax weights. Scores are in log2 units; the
// warp's online-softmax state st is updated in place. Shared-memory reads
// are conflict-free: each K or V row is read whole by consecutive lanes
// (odd rows with their two 16-byte halves swapped), q and the weights by
// groups of lanes at one address.
template <int HD, int G>
__device__ __forceinline__ void attn_chunk(AttnWarpState<HD, G> &st, const uint16_t *Kp,
                                           const uint16_t *Vp, int npos, const float *q,
                                           float *pbuf) {
    using Lay = AttnLayout<HD, G>;
    constexpr int DQ = Lay::DQ, PG = Lay::PG, NPASS = Lay::NPASS, DGV = Lay::DGV, PGV = Lay::PGV;
    constexpr int GP = Lay::GP;
    const int lane = threadIdx.x & 31;
    const int pl = lane / DQ, dq = lane % DQ;
    // ---- scores of head dq % GP at positions k*PG + pl
    float s[NPASS];
    {
        float2 qr[GP][8];
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            const float4 *qg = reinterpret_cast<const float4 *>(q + Lay::qidx(g < G ? g : 0, dq * 16));
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float4 v = g < G ? qg[c] : make_float4(0.f, 0.f, 0.f, 0.f);
                qr[g][2 * c] = make_float2(v.x, v.y);
                qr[g][2 * c + 1] = make_float2(v.z, v.w);
            }
        }
#pragma unroll
        for (int k = 0; k < NPASS; ++k) {
            const int pos = k * PG + pl;
            const bool valid = pos < npos;
            const int row = valid ? pos : 0;
            // 32 bytes of this row: halves in an order that depends on the
            // row's bank offset so that a pass touches every bank evenly
            const bool swap = ((row + (dq * 32) / 128) & 1) != 0;
            const uint4 *kr = reinterpret_cast<const uint4 *>(Kp + (size_t)row * HD + dq * 16);
            uint4 w0 = kr[swap ? 1 : 0], w1 = kr[swap ? 0 : 1];
            if (swap) {
                const uint4 t = w0;
                w0 = w1;
                w1 = t;
            }
            const uint32_t u[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
            float v[GP];
#pragma unroll
            for (int g = 0; g < GP; ++g) {
                float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    a = __ffma2_rn(make_float2(bf_lo(u[e]), bf_hi(u[e])), qr[g][e], a);
                    b = __ffma2_rn(make_float2(bf_lo(u[e + 1]), bf_hi(u[e + 1])), qr[g][e + 1], b);
                }
                v[g] = (a.x + a.y) + (b.x + b.y);
            }
            // reduce-scatter over the low dim-group bits, then plain sums
            float c;
            if constexpr (GP == 4) {
                const bool hi2 = (dq & 2) != 0, hi1 = (dq & 1) != 0;
                float a0 = hi2 ? v[2] : v[0], a1 = hi2 ? v[3] : v[1];
                const float b0 = hi2 ? v[0] : v[2], b1 = hi2 ? v[1] : v[3];
                a0 += __shfl_xor_sync(0xFFFFFFFFu, b0, 2);
                a1 += __shfl_xor_sync(0xFFFFFFFFu, b1, 2);
                c = hi1 ? a1 : a0;
                c += __shfl_xor_sync(0xFFFFFFFFu, hi1 ? a0 : a1, 1);
#pragma unroll
                for (int o = 4; o < DQ; o <<= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
            } else if constexpr (GP == 2) {
                const bool hi1 = (dq & 1) != 0;
                c = hi1 ? v[1] : v[0];
                c += __shfl_xor_sync(0xFFFFFFFFu, hi1 ? v[0] : v[1], 1);
#pragma unroll
                for (int o = 2; o < DQ; o <<= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
            } else {
                c = v[0];
#pragma unroll
                for (int o = 1; o < DQ; o <<= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
            }
            s[k] = valid ? c : -INFINITY;
        }
    }
    // ---- online softmax of this lane's head across the chunk; positions
    // differ in the lane bits above the dim group
    const int hg = dq % GP;
    float mloc = s[0];
#pragma unroll
    for (int k = 1; k < NPASS; ++k) mloc = fmaxf(mloc, s[k]);
#pragma unroll
    for (int o = DQ; o < 32; o <<= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xFFFFFFFFu, mloc, o));
    const float mnew = fmaxf(st.m, mloc);
    const float corr = exp2f(st.m - mnew);
    float ls = 0.f;
#pragma unroll
    for (int k = 0; k < NPASS; ++k) {
        s[k] = exp2f(s[k] - mnew);  // exp2(-inf) = 0 for invalid positions
        ls += s[k];
    }
#pragma unroll
    for (int o = DQ; o < 32; o <<= 1) ls += __shfl_xor_sync(0xFFFFFFFFu, ls, o);
    st.l = st.l * corr + ls;
    st.m = mnew;
    if (dq < GP && hg < G) {
#pragma unroll
        for (int k = 0; k < NPASS; ++k) pbuf[(k * PG + pl) * 4 + hg] = s[k];
    }
    // every lane rescales all heads: head g's factor from lane g (pl 0, dq g)
    float cg[G];
#pragma unroll
    for (int g = 0; g < G; ++g) cg[g] = __shfl_sync(0xFFFFFFFFu, corr, g);
    __syncwarp();
    // ---- P.V
    {
        const int pv = lane / DGV, dg = lane % DGV;
        float2 o2[G][4];
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                o2[g][e] = make_float2(st.o[g][2 * e] * cg[g], st.o[g][2 * e + 1] * cg[g]);
#pragma unroll
        for (int i = 0; i < 32 / PGV; ++i) {
            const int pos = i * PGV + pv;
            if (pos < npos) {
                const float4 pp = *reinterpret_cast<const float4 *>(pbuf + pos * 4);
                const uint4 w = *reinterpret_cast<const uint4 *>(Vp + (size_t)pos * HD + dg * 8);
                const uint32_t u[4] = {w.x, w.y, w.z, w.w};
                const float pg[4] = {pp.x, pp.y, pp.z, pp.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 v = make_float2(bf_lo(u[e]), bf_hi(u[e]));
#pragma unroll
                    for (int g = 0; g < G; ++g) o2[g][e] = __ffma2_rn(v, make_float2(pg[g], pg[g]), o2[g][e]);
                }
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                st.o[g][2 * e] = o2[g][e].x;
                st.o[g][2 * e + 1] = o2[g][e].y;
            }
    }
    __syncwarp();
}

template <int HD, int G>
__device__ void do_attn_hd(const Params &p, const Ctx &cx, const Instr &in, uint32_t &t, bool &bad) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int l = in.layer, kvh = in.a0, split = in.a1;
    const int gq0 = kvh * p.G + in.slot * G;  // first query head of this instruction
    const int b = seq_of(p, in), pos = pos_of(p, b);  // sequence of a batched step
    const AttnRange r = attn_range(p, split, pos);
    const int seff = attn_seff(p, pos);
    if (!r.active) return;  // nothing cached for this split at this position
    const uint32_t ep8 = cx.misc->ep8;
    if (tid == 0) cx.misc->staged_key = -1;  // xbuf becomes attention scratch
    const int qkv_stride = (p.Hq + 2 * p.Hkv) * HD;
    const uint2 *qkv = p.qkvll + ((size_t)l * p.nb + b) * qkv_stride;
    // shared scratch: q [G][QSTR] | knew [HD] bf16 | vnew [HD] bf16 | warp states
    // [8][G][HD+4]; the host checks G*QSTR + HD + 8*G*(HD+4) <= kXbufFloats.
    using Lay = AttnLayout<HD, G>;
    float *qs = cx.xbuf;
    uint16_t *knew = reinterpret_cast<uint16_t *>(cx.xbuf + G * Lay::QSTR);
    uint16_t *vnew = knew + HD;
    constexpr int WS = HD + 4;  // warp-state row: HD outputs, max, sum, pad (16-byte rows)
    float *wst = cx.xbuf + G * Lay::QSTR + HD;
    float *pbuf = cx.red + warp * (32 * kMaxG);

    // q of the group's heads (rotated, pre-scaled by log2(e)/sqrt(hd)) and,
    // for the split that owns the new position, its key and value: polled
    // from the QKV instructions' tagged outputs.
    {
        const float qscale = 1.4426950408889634f / sqrtf((float)HD);
        const float *rope = p.rope + (size_t)pos * HD;  // [HD/2][2]
        for (int idx = tid; idx < G * (HD / 2); idx += kConsumerThreads) {
            const int g = idx / (HD / 2), i = idx % (HD / 2);
            const uint2 *qh = qkv + (size_t)(gq0 + g) * HD;
            const uint2 *srcs[2] = {qh + i, qh + i + HD / 2};
            float ab[2];
            if (bad || !ll_read_n<2>(p, srcs, ep8, ab) || !CHK(rope + 2 * i, 8, 28) ||
                !CHKS(qs + Lay::qidx(g, i + HD / 2), 4, 48)) {
                bad = true;
                continue;
            }
            const float a = ab[0], b = ab[1];
            const float c = rope[2 * i], s = rope[2 * i + 1];
            qs[Lay::qidx(g, i)] = (a * c - b * s) * qscale;
            qs[Lay::qidx(g, i + HD / 2)] = (b * c + a * s) * qscale;
        }
        if (r.has_new) {
            const uint2 *kh = qkv + (size_t)p.Hq * HD + (size_t)kvh * HD;
            const uint2 *vh = qkv + (size_t)(p.Hq + p.Hkv) * HD + (size_t)kvh * HD;
            const size_t cache_off = (((size_t)l * p.max_batch + slot_of(p, b)) * p.Hkv + kvh) * p.max_seq * HD +
                                     (size_t)pos * HD;
            for (int i = tid; i < HD / 2; i += kConsumerThreads) {
                const uint2 *srcs[4] = {kh + i, kh + i + HD / 2, vh + i, vh + i + HD / 2};
                float kv4[4];
                if (bad || !ll_read_n<4>(p, srcs, ep8, kv4) || !CHK(p.kc + cache_off + i, 2, 24) || !CHK(p.kc + cache_off + i + HD / 2, 2, 24) ||
                    !CHK(p.vc + cache_off + i, 2, 24) || !CHK(p.vc + cache_off + i + HD / 2, 2, 24) ||
                    !CHK(rope + 2 * i, 8, 28) || !CHKS(vnew + i + HD / 2, 2, 49)) {
                    bad = true;
                    continue;
                }
                const float a = kv4[0], b = kv4[1];
                const float c = rope[2 * i], s = rope[2 * i + 1];
                const uint16_t k0 = f2bf(a * c - b * s), k1 = f2bf(b * c + a * s);
                const uint16_t v0 = f2bf(kv4[2]), v1 = f2bf(kv4[3]);
                knew[i] = k0;
                knew[i + HD / 2] = k1;
                vnew[i] = v0;
                vnew[i + HD / 2] = v1;
                if (in.slot == 0) {  // one instruction of the kv head appends to the cache
                    p.kc[cache_off + i] = k0;
                    p.kc[cache_off + i + HD / 2] = k1;
                    p.vc[cache_off + i] = v0;
                    p.vc[cache_off + i + HD / 2] = v1;
                }
            }
        }
        bad = consumer_sync_any(bad);
        phase_stamp(p, cx, 0);
    }
    // per-warp online softmax over the split's tiles
    AttnWarpState<HD, G> st;
    st.m = -INFINITY;
    st.l = 0.f;
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < 8; ++e) st.o[g][e] = 0.f;
    // Tiles of ppt positions are split into chunks of 32 (one lane per
    // position); tile j goes to warp group j % slots, chunk c of it to warp
    // group_base + c, so the chunks of a short context run side by side.
    constexpr int CPT = (kPageBytes / 2) / (HD * 2) / 32;  // chunks per tile
    constexpr int SLOTS = kConsumerWarps / CPT;
    // the new position needs only the polled q/k/v: the last warp does it
    // while the cached tiles may still be landing
    if (!bad && r.has_new && warp == kConsumerWarps - 1) attn_chunk<HD, G>(st, knew, vnew, 1, qs, pbuf);
    const int nt = (r.t1 - r.t0 + p.ppt - 1) / p.ppt;
    for (int j = 0; j < nt; ++j, ++t) {
        const int pg = t % kPages;
        if (!bad && !wait_tile(p, cx, pg, (t / kPages) & 1, p.trace != nullptr)) bad = true;
        const int chunk = warp - (j % SLOTS) * CPT;
        if (!bad && chunk >= 0 && chunk < CPT) {
            const int ts = r.t0 + j * p.ppt;
            int n = r.t1 - ts;
            if (n > p.ppt) n = p.ppt;
            int np = n - chunk * 32;
            np = np > 32 ? 32 : np;
            if (np > 0 && CHKS(cx.pages + (size_t)pg * kPageBytes + (size_t)(chunk * 32 + np) * HD * 2 - 2, 2, 50) &&
                CHKS(pbuf + 32 * kMaxG - 1, 4, 51)) {
                const uint16_t *Kp = reinterpret_cast<const uint16_t *>(cx.pages + (size_t)pg * kPageBytes) +
                                     (size_t)chunk * 32 * HD;
                const uint16_t *Vp = reinterpret_cast<const uint16_t *>(cx.pages + (size_t)pg * kPageBytes +
                                                                          kPageBytes / 2) +
                                     (size_t)chunk * 32 * HD;
                attn_chunk<HD, G>(st, Kp, Vp, np, qs, pbuf);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&cx.empty[pg]);
    }
    bad = consumer_sync_any(bad);
    phase_stamp(p, cx, 1);
    if (bad) return;
    // warp states -> shared: sum the P.V lanes' position groups, then the
    // lanes of group 0 hold the warp's output dims dg*8 .. dg*8+7; lane g
    // (position 0, dim group g of the score layout) holds head g's max and sum
    {
        constexpr int DGV = AttnLayout<HD, G>::DGV;
        float *my = wst + (size_t)warp * G * WS;
        if (!CHKS(my + G * WS - 1, 4, 52)) my = wst;
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < 8; ++e)
#pragma unroll
                for (int o = DGV; o < 32; o <<= 1) st.o[g][e] += __shfl_xor_sync(0xFFFFFFFFu, st.o[g][e], o);
        if (lane < DGV) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float4 *dst = reinterpret_cast<float4 *>(my + g * WS + lane * 8);
                dst[0] = make_float4(st.o[g][0], st.o[g][1], st.o[g][2], st.o[g][3]);
                dst[1] = make_float4(st.o[g][4], st.o[g][5], st.o[g][6], st.o[g][7]);
            }
        }
        if (lane < G) {
            my[lane * WS + HD] = st.m;
            my[lane * WS + HD + 1] = st.l;
        }
    }
    consumer_sync();
    // output word of element idx of this kv group's heads (batched steps: interleaved)
    // (batched steps: plain fp32, interleaved, released by the attn_done counter)
    uint2 *const out = p.attll + (size_t)l * p.Hq * HD + (size_t)gq0 * HD;
    float *const outf = reinterpret_cast<float *>(p.attll) + (size_t)l * kMaxBatch * p.Hq * HD;
    auto put = [&](int idx, float v) {
        if (p.nb > 1) {
            float *dst = outf + bofs(b, gq0 * HD + idx);
            if (CHK(dst, 4, 27)) *dst = v;
        } else if (CHK(out + idx, 8, 27)) {
            ll_store(out + idx, v, ep8);
        }
    };
    if (seff == 1) {
        // The only active split holds the whole context: normalise and
        // publish the attention output directly.
        for (int idx = tid; idx < G * HD; idx += kConsumerThreads) {
            const int g = idx / HD, e = idx % HD;
            float M = -INFINITY;
            for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, wst[(w * G + g) * WS + HD]);
            float num = 0.f, den = 0.f;
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float mw = wst[(w * G + g) * WS + HD];
                if (mw == -INFINITY) continue;
                const float wgt = exp2f(mw - M);
                num += wst[(w * G + g) * WS + e] * wgt;
                den += wst[(w * G + g) * WS + HD + 1] * wgt;
            }
            put(idx, num / den);
        }
        if (p.nb > 1) {  // batched steps: release this (sequence, kv head)'s output
            consumer_sync();
            if (tid == 0) ctr_signal(p, p.cl.attn_done + l, 1);
        }
        return;
    }
    // Several splits: publish this split's partial (o unnormalised, m, l) ...
    constexpr int PS = HD + 2;  // partial row in global memory: HD outputs, max, sum
    uint2 *part = p.partll + (((size_t)l * p.nb + b) * p.Hq + (size_t)gq0) * p.S * PS;
    for (int idx = tid; idx < G * PS; idx += kConsumerThreads) {
        const int g = idx / PS, e = idx % PS;
        float M = -INFINITY;
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, wst[(w * G + g) * WS + HD]);
        float acc = 0.f;
        if (e == HD) {
            acc = M;
        } else if (M != -INFINITY) {
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float mw = wst[(w * G + g) * WS + HD];
                if (mw != -INFINITY) acc += wst[(w * G + g) * WS + e] * exp2f(mw - M);
            }
        }
        uint2 *dst = part + ((size_t)g * p.S + split) * PS + e;
        if (CHK(dst, 8, 25)) ll_store(dst, acc, ep8);
    }
    // ... and the split that owns the new position merges all of them
    // (log-sum-exp), polling the others' tagged partials with all loads of
    // a poll in flight together.
    if (!r.has_new) return;
    for (int idx = tid; idx < G * HD && !bad; idx += kConsumerThreads) {
        const int g = idx / HD, e = idx % HD;
        const uint2 *sg = part + (size_t)g * p.S * PS;
        float num = 0.f, den = 0.f, M = -INFINITY;
        for (int s0 = 0; s0 < seff && !bad; s0 += kMergeBatch) {
            const int ns = seff - s0 < kMergeBatch ? seff - s0 : kMergeBatch;
            uint2 mv[kMergeBatch], lv[kMergeBatch], ov[kMergeBatch];
            Spin sp;
            while (true) {
                bool ok = true;
#pragma unroll
                for (int k = 0; k < kMergeBatch; ++k) {
                    if (k < ns) {
                        const uint2 *ps = sg + (size_t)(s0 + k) * PS;
                        mv[k] = ll_ld8(ps + HD);
                        lv[k] = ll_ld8(ps + HD + 1);
                        ov[k] = ll_ld8(ps + e);
                    }
                }
#pragma unroll
                for (int k = 0; k < kMergeBatch; ++k)
                    if (k < ns) ok = ok && mv[k].y == ep8 && lv[k].y == ep8 && ov[k].y == ep8;
                if (ok) break;
                if (!sp.keep_going(p)) {
                    bad = true;
                    break;
                }
            }
            if (bad) break;
            // online combination across batches of splits
#pragma unroll
            for (int k = 0; k < kMergeBatch; ++k) {
                if (k >= ns) continue;
                const float m = __uint_as_float(mv[k].x);
                if (m == -INFINITY) continue;
                const float Mn = fmaxf(M, m);
                const float a = exp2f(M - Mn), b = exp2f(m - Mn);
                num = num * a + __uint_as_float(ov[k].x) * b;
                den = den * a + __uint_as_float(lv[k].x) * b;
                M = Mn;
            }
        }
        if (!bad) put(idx, num / den);
    }
    bad = consumer_sync_any(bad);
    if (p.nb > 1 && !bad && tid == 0) ctr_signal(p, p.cl.attn_done + l, 1);
}

// ---------------------------------------------------------------------------
// Consumer: interprets the queue.
// ---------------------------------------------------------------------------
template <int HD, int G, bool BATCH>
__device__ void consumer(const Params &p, const Ctx &cx, int qb, int qe, int q0) {
    const int tid = threadIdx.x;
    uint32_t t = 0;
    bool bad = false;
    long long *trace = p.trace ? p.trace + (size_t)blockIdx.x * p.trace_cap * kTraceWords : nullptr;
    for (int i = qb; i < qe && !bad; ++i) {
        const Instr in = load_instr(p, i);
        if (i + 1 < qe) prefetch_instr(p, i + 1);
        const uint64_t ts = trace ? gtimer() : 0;
        if (trace && tid == 0) {
            cx.misc->phase[0] = cx.misc->phase[1] = cx.misc->phase[2] = (long long)ts;
            cx.misc->tile_wait = 0;
        }
        if (in.op == OP_ATTN) {
            do_attn_hd<HD, G>(p, cx, in, t, bad);
        } else if constexpr (BATCH) {
            gemv_batch(p, cx, in, t, bad);
            if (tid == 0) cx.misc->staged_key = -1;
        } else {
            do_gemv(p, cx, in, t, bad);
        }
        phase_stamp(p, cx, 2);
        bad = consumer_sync_any(bad);
        if (bad) break;
        if (tid == 0 && trace && (i - q0) < p.trace_cap &&
            CHK(trace + (size_t)(i - q0) * kTraceWords, 8 * kTraceWords, 34)) {
            long long *rec = trace + (size_t)(i - q0) * kTraceWords;  // slot = place in the SM's queue
            rec[0] = blockIdx.x;
            rec[1] = in.op;
            rec[2] = (long long)ts - cx.misc->tile_wait;  // start minus time spent waiting for tiles
            rec[3] = (long long)ts;
            rec[4] = cx.misc->phase[0];
            rec[5] = cx.misc->phase[1];
            rec[6] = cx.misc->phase[2];
            rec[7] = (long long)gtimer();
        }
    }
    if (bad && tid == 0) cx.misc->aborted = 1;
}

// The kernel is instantiated per head dimension and per group size G
// (query heads per kv head) so that each instance holds only the attention
// code its model runs: a smaller instruction footprint keeps the hot loops
// in the instruction cache. BATCH instances run batched steps (nb > 1); the
// single-sequence instances carry none of that code.
template <int HD, int G, bool BATCH>
__global__ void __launch_bounds__(kThreads, 1) mk_megakernel(const Params prm) {
    uint8_t *smem = mk_smem;
    // Launch parameters are copied to shared memory once; every device
    // function reads them from there (no generic pointer into param space).
    Params *sp = reinterpret_cast<Params *>(smem + kSmemParams);
    Ctx cx;
    cx.pages = smem + kSmemPages;
    cx.xbuf = reinterpret_cast<float *>(smem + kSmemXbuf);
    cx.red = reinterpret_cast<float *>(smem + kSmemRed);
    cx.resid = reinterpret_cast<float *>(smem + kSmemResid);
    cx.dred = reinterpret_cast<float *>(smem + kSmemDred);
    cx.full = reinterpret_cast<uint64_t *>(smem + kSmemBars);
    cx.empty = cx.full + kPages;
    cx.misc = reinterpret_cast<Misc *>(smem + kSmemMisc);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        *sp = prm;
        for (int i = 0; i < kPages; ++i) {
            mbar_init(&cx.full[i], 1);
            mbar_init(&cx.empty[i], kConsumerWarps);
        }
        cx.misc->flag = 0;
        cx.misc->polling = 0;
        cx.misc->aborted = 0;
        cx.misc->n_issued = 0;
        cx.misc->staged_key = -1;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    const Params &p = *sp;
    if (tid == 0) {
        // positions held in device memory are read once, before anything uses them
        if (p.d_pos) {
            for (int b = 0; b < p.nb && b < kMaxBatch; ++b)
                sp->posb[b] = CHK(p.d_pos + b, 4, 33) ? *(volatile const int32_t *)(p.d_pos + b) : -1;
            sp->pos = sp->posb[0];
        }
        // a single sequence's token held in memory is read once as well (it
        // may sit in host memory; the last CTA may overwrite it at the end)
        if (p.d_token && p.nb <= 1) {
            sp->token = CHK(p.d_token, 4, 33) ? *(volatile const int32_t *)p.d_token : -1;
            sp->d_token = nullptr;
        }
        uint32_t e = 1;
        if (CHK(p.epoch, 4, 32)) e = *(volatile uint32_t *)p.epoch & 0xFFFFFFu;
        cx.misc->ep8 = (e ? e : 1u) << 8;
    }
    __syncthreads();
    const int *qrow = p.q_begin + (size_t)blockIdx.x * (p.n_stages + 1);
    bool run = CHK(qrow + p.stage_lo, 4, 2) && CHK(qrow + p.stage_hi, 4, 2) &&
               CHK(p.status, 4, 32) && CHK(p.abort_flag, 4, 32) && CHK(p.exit_ctr, 4, 32);
    const int qb = run ? __ldg(qrow + p.stage_lo) : 0, qe = run ? __ldg(qrow + p.stage_hi) : 0;
    const int q0 = run ? __ldg(qrow) : 0;  // the SM's first instruction (trace slots)
    run = run && *(volatile int32_t *)p.status == DS_OK;
    if (run) {
        bool bad_tok = false, bad_pos = false;
        for (int b = 0; b < p.nb; ++b) {
            const int tok = current_token(p, b), pos = pos_of(p, b);
            bad_tok = bad_tok || tok < 0 || tok >= p.V;
            bad_pos = bad_pos || pos < 0 || pos >= p.max_seq;
        }
        if (bad_tok || bad_pos) {
            if (tid == 0) {
                atomicCAS(p.status, DS_OK, bad_tok ? DS_BAD_TOKEN : DS_BAD_POS);
                atomicExch(p.abort_flag, 1);
            }
            run = false;
        }
    }
    if (run) {
        if (warp == kConsumerWarps) {
            producer(p, cx, qb, qe);
        } else {
            consumer<HD, G, BATCH>(p, cx, qb, qe, q0);
        }
    }
    __syncthreads();
    // Drain: copies issued but never consumed (only after an abort) must land
    // before the CTA's shared memory is released.
    if (tid == 0 && run) {
        const uint32_t ni = cx.misc->n_issued;
        const uint32_t lo = ni > (uint32_t)kPages ? ni - kPages : 0u;
        for (uint32_t t = lo; t < ni; ++t) {
            const uint64_t t0 = gtimer();
            while (!mbar_try_wait(&cx.full[t % kPages], (t / kPages) & 1)) {
                if (gtimer() - t0 > 1000000000ull) break;
            }
        }
    }
    // End of step: the last CTA out resets the counters and advances the
    // epoch that tags this step's activations.
    if (p.reset_at_exit && tid == 0 && CHK(p.exit_ctr, 4, 32) &&
        CHK(p.ctr + p.cl.total - 1, 4, 32) && CHK(p.epoch, 4, 32)) {
        __threadfence();
        const uint32_t old = atomicAdd(p.exit_ctr, 1u);
        if (old == gridDim.x - 1) {
            __threadfence();
            for (int c = 0; c < p.cl.total; ++c) p.ctr[c] = 0u;
            const uint32_t e = (cx.misc->ep8 >> 8) + 1u;
            *(volatile uint32_t *)p.epoch = (e & 0xFFFFFFu) ? (e & 0xFFFFFFu) : 1u;
            *p.abort_flag = 0;
            *p.exit_ctr = 0u;
            __threadfence();
        }
    }
}

}  // namespace
}  // namespace mk
