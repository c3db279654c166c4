// mk_kernel.cu — the persistent decode megakernel (sm_103a).
//
// One CTA per SM interprets that SM's instruction queue (planned on the host,
// see mk_host.cpp). The design is the one described in "Revolution der
// KI-Beschleunigung: Wie ein Low-Latency Megakernel den Llama-1B Turbo
// zündet" (dasgeld.co), rebuilt for GB300:
//   * the whole decode step is one launch; stages that used to be separate
//     kernels are instructions (megakernel paragraphs);
//   * instructions wait on and bump dependency counters in global memory,
//     per kv-head group for attention (synchronisation paragraph);
//   * shared memory is a ring of pages: a producer warp streams the next
//     instructions' weights (and cached keys/values) into free pages with
//     cp.async.bulk while the consumer warps compute, across dependency
//     waits, so HBM keeps streaming during synchronisation (shared-memory
//     paging paragraph);
//   * bf16 weights, fp32 accumulation (latency paragraph).
//
// CTA layout: warps 0..7 are consumers (GEMV / attention math), warp 8 lane 0
// is the producer that issues bulk copies. Page p has a "full" mbarrier
// (producer -> consumers, completed by the copy's transaction bytes) and an
// "empty" mbarrier (8 consumer warps -> producer).
//
// Every wait is bounded (%globaltimer): on expiry the CTA records a timeout
// in the status word, raises the abort flag that all CTAs poll, waits for
// its own copies in flight and returns. Nothing traps.
#include <cuda_runtime.h>
#include <stdint.h>

#include "mk_plan.h"

namespace mk {

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
extern __shared__ __align__(1024) uint8_t mk_smem[];

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
        a + bytes <= (uintptr_t)(p.trace + (size_t)gridDim.x * p.trace_cap * 5))
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

// Orderable key for the argmax: larger value wins, then lower index.
__device__ __forceinline__ unsigned long long argmax_key(float v, uint32_t idx) {
    uint32_t u = __float_as_uint(v);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return (static_cast<unsigned long long>(u) << 32) | (0xFFFFFFFFu - idx);
}

// ---------------------------------------------------------------------------
// Shared state
// ---------------------------------------------------------------------------
struct Misc {
    float red8[kConsumerWarps];
    unsigned long long best8[kConsumerWarps];
    volatile int32_t flag;      // broadcast slot (wait result / last-arrival)
    volatile int32_t aborted;   // this CTA gave up
    volatile uint32_t n_issued; // tiles issued by the producer
    int32_t pad;
};

struct Ctx {
    uint8_t *pages;
    float *xbuf;
    float *red;
    uint64_t *full, *empty;
    Misc *misc;
};

// Bounded spin of one thread on a global counter. Returns false on abort or
// timeout (after recording the timeout).
__device__ bool wait_counter(const Params &p, const uint32_t *c, uint32_t target) {
    if (!CHK(c, 4, 29)) return false;
    if (ld_acquire(c) >= target) return true;
    uint64_t t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        if (ld_acquire(c) >= target) return true;
        if ((it & 31u) == 0) {
            if (*(volatile int32_t *)p.abort_flag) return false;
            if (gtimer() - t0 > p.timeout_ns) {
                atomicCAS(p.status, DS_OK, DS_TIMEOUT);
                atomicExch(p.abort_flag, 1);
                return false;
            }
        }
    }
}

// Bounded wait on an mbarrier phase.
__device__ bool wait_bar(const Params &p, uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*(volatile int32_t *)p.abort_flag) return false;
            if (gtimer() - t0 > p.timeout_ns) {
                atomicCAS(p.status, DS_OK, DS_TIMEOUT);
                atomicExch(p.abort_flag, 1);
                return false;
            }
        }
    }
}

__device__ __forceinline__ Instr load_instr(const Params &p, int i) {
    Instr in;
    if (!CHK(p.instr + i, sizeof(Instr), 1)) {
        memset(&in, 0, sizeof in);
        in.wait_ctr = -1;
        in.op = OP_QKV;
        in.a1 = 0;
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

// ---------------------------------------------------------------------------
// Attention split bookkeeping (identical on producer and consumer side).
// Cached positions [0, pos) are cut into seff <= S contiguous chunks of at
// least one tile; the last active split also owns the new position `pos`.
// ---------------------------------------------------------------------------
struct AttnRange {
    int active, t0, t1, has_new;
};

__device__ __forceinline__ int attn_seff(const Params &p) {
    int need = (p.pos + p.ppt - 1) / p.ppt;
    if (need < 1) need = 1;
    return need < p.S ? need : p.S;
}

__device__ __forceinline__ AttnRange attn_range(const Params &p, int split) {
    AttnRange r;
    int seff = attn_seff(p);
    r.active = split < seff;
    int chunk = (p.pos + seff - 1) / seff;
    r.t0 = split * chunk;
    if (r.t0 > p.pos) r.t0 = p.pos;
    r.t1 = r.t0 + chunk;
    if (r.t1 > p.pos) r.t1 = p.pos;
    r.has_new = (split == seff - 1);
    return r;
}

__device__ __forceinline__ int num_tiles(const Params &p, const Instr &in) {
    if (in.op == OP_ATTN) {
        AttnRange r = attn_range(p, in.a1);
        if (!r.active) return 0;
        return (r.t1 - r.t0 + p.ppt - 1) / p.ppt;
    }
    const Geo &g = geo_of(p, in.op);
    int per = (in.op == OP_GATEUP) ? g.rt / 2 : g.rt;
    return (in.a1 + per - 1) / per;
}

// ---------------------------------------------------------------------------
// Producer: walks the same queue and issues every tile into the page ring.
// ---------------------------------------------------------------------------
__device__ void producer(const Params &p, const Ctx &cx, int qb, int qe) {
    const uint64_t pol = policy_evict_first();
    uint32_t t = 0;
    for (int i = qb; i < qe; ++i) {
        const Instr in = load_instr(p, i);
        const int nt = num_tiles(p, in);
        for (int j = 0; j < nt; ++j, ++t) {
            const int pg = t % kPages;
            if (t >= kPages && !wait_bar(p, &cx.empty[pg], ((t / kPages) - 1) & 1)) {
                cx.misc->aborted = 1;
                return;
            }
            uint8_t *dst = cx.pages + (size_t)pg * kPageBytes;
            if (in.op == OP_ATTN) {
                AttnRange r = attn_range(p, in.a1);
                int ts = r.t0 + j * p.ppt;
                int n = r.t1 - ts;
                if (n > p.ppt) n = p.ppt;
                size_t base = ((size_t)(in.layer * p.max_batch) * p.Hkv + in.a0) * p.max_seq * p.hd +
                              (size_t)ts * p.hd;
                uint32_t bytes = (uint32_t)n * p.hd * 2;
                const bool ok = CHK(p.kc + base, bytes, 3) && CHK(p.vc + base, bytes, 4) &&
                                CHKS(dst, kPageBytes / 2 + bytes, 40);
                mbar_expect_tx(&cx.full[pg], ok ? 2 * bytes : 0);
                if (ok) {
                    bulk_g2s(dst, p.kc + base, bytes, &cx.full[pg], pol);
                    bulk_g2s(dst + kPageBytes / 2, p.vc + base, bytes, &cx.full[pg], pol);
                }
            } else {
                const Geo &g = geo_of(p, in.op);
                const int per = (in.op == OP_GATEUP) ? g.rt / 2 : g.rt;
                int rows = in.a1 - j * per;
                if (rows > per) rows = per;
                const size_t row0 = (size_t)in.a0 + (size_t)j * per;
                const uint32_t bytes = (uint32_t)rows * g.K * 2;
                if (in.op == OP_GATEUP) {
                    const LayerW *lw = p.layers + in.layer;
                    const bool ok = CHK(lw->w_gate + row0 * g.K, bytes, 5) &&
                                    CHK(lw->w_up + row0 * g.K, bytes, 6) &&
                                    CHKS(dst, (size_t)per * g.K * 2 + bytes, 41);
                    mbar_expect_tx(&cx.full[pg], ok ? 2 * bytes : 0);
                    if (ok) {
                        bulk_g2s(dst, lw->w_gate + row0 * g.K, bytes, &cx.full[pg], pol);
                        bulk_g2s(dst + (size_t)per * g.K * 2, lw->w_up + row0 * g.K, bytes,
                                 &cx.full[pg], pol);
                    }
                } else {
                    const uint16_t *W;
                    const LayerW *lw = p.layers + in.layer;
                    switch (in.op) {
                        case OP_QKV: W = in.mat == 0 ? lw->wq : (in.mat == 1 ? lw->wk : lw->wv); break;
                        case OP_OPROJ: W = lw->wo; break;
                        case OP_DOWN: W = lw->w_down; break;
                        default: W = p.embed; break;
                    }
                    const bool ok = CHK(W + row0 * g.K, bytes, 7) && CHKS(dst, bytes, 42);
                    mbar_expect_tx(&cx.full[pg], ok ? bytes : 0);
                    if (ok) bulk_g2s(dst, W + row0 * g.K, bytes, &cx.full[pg], pol);
                }
            }
            cx.misc->n_issued = t + 1;
        }
    }
}

// ---------------------------------------------------------------------------
// GEMV instructions
// ---------------------------------------------------------------------------

// Dot product of one warp-slice of a bf16 row (in shared memory) with the
// lane's nx input floats. Element e of chunk c of this lane is input index
// (c*32 + lane)*8 + e of the slice.
template <int NX>
__device__ __forceinline__ float dot_row(const uint4 *w, const float *xr) {
    uint4 wv[NX / 8];
#pragma unroll
    for (int c = 0; c < NX / 8; ++c) wv[c] = w[c * 32];
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int c = 0; c < NX / 8; ++c) {
        const float *x = xr + c * 8;
        a0 = fmaf(bf_lo(wv[c].x), x[0], a0);
        a1 = fmaf(bf_lo(wv[c].y), x[2], a1);
        a2 = fmaf(bf_lo(wv[c].z), x[4], a2);
        a3 = fmaf(bf_lo(wv[c].w), x[6], a3);
        a0 = fmaf(bf_hi(wv[c].x), x[1], a0);
        a1 = fmaf(bf_hi(wv[c].y), x[3], a1);
        a2 = fmaf(bf_hi(wv[c].z), x[5], a2);
        a3 = fmaf(bf_hi(wv[c].w), x[7], a3);
    }
    return (a0 + a1) + (a2 + a3);
}

// Runs every tile of a GEMV instruction: per-row partial dot products go to
// red[out_index * sw + ks]. `xsrc` is the input vector (shared memory when
// staged, global memory otherwise).
template <int NX>
__device__ void gemv_tiles(const Params &p, const Ctx &cx, const Instr &in, const Geo &g,
                           const float *xsrc, bool xglobal, uint32_t &t, bool &bad) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rg = warp / g.sw, ks = warp % g.sw;
    // this lane's input slice
    float xr[NX];
    const int sbase = ks * g.kslice;
#pragma unroll
    for (int c = 0; c < NX / 8; ++c) {
        const int idx = sbase + (c * 32 + lane) * 8;
        float4 u = make_float4(0.f, 0.f, 0.f, 0.f), v = u;
        if (xglobal) {
            if (CHK(xsrc + idx, 32, 8)) {
                u = __ldcg(reinterpret_cast<const float4 *>(xsrc + idx));
                v = __ldcg(reinterpret_cast<const float4 *>(xsrc + idx + 4));
            }
        } else if (CHKS(xsrc + idx, 32, 43)) {
            u = *reinterpret_cast<const float4 *>(xsrc + idx);
            v = *reinterpret_cast<const float4 *>(xsrc + idx + 4);
        }
        xr[c * 8 + 0] = u.x; xr[c * 8 + 1] = u.y; xr[c * 8 + 2] = u.z; xr[c * 8 + 3] = u.w;
        xr[c * 8 + 4] = v.x; xr[c * 8 + 5] = v.y; xr[c * 8 + 6] = v.z; xr[c * 8 + 7] = v.w;
    }
    const bool gu = in.op == OP_GATEUP;
    const int n = in.a1;
    const int per = gu ? g.rt / 2 : g.rt;
    const int nt = (n + per - 1) / per;
    const size_t row_bytes = (size_t)g.K * 2;
    for (int j = 0; j < nt; ++j, ++t) {
        const int pg = t % kPages;
        if (!bad && !wait_bar(p, &cx.full[pg], (t / kPages) & 1)) bad = true;
        if (!bad) {
            const uint8_t *page = cx.pages + (size_t)pg * kPageBytes;
            for (int mi = 0; mi < g.m; ++mi) {
                const int r = rg * g.m + mi;  // row of the tile
                int out_i;
                bool valid;
                if (gu) {
                    const int up = r >= per;
                    const int rr = j * per + (up ? r - per : r);
                    valid = rr < n;
                    out_i = up ? n + rr : rr;
                } else {
                    out_i = j * per + r;
                    valid = out_i < n;
                }
                if (valid) {
                    const uint4 *w = reinterpret_cast<const uint4 *>(page + r * row_bytes) +
                                     (sbase / 8) + lane;
                    const bool ok = CHKS(w, 16, 44) && CHKS(w + (NX / 8 - 1) * 32, 16, 45);
                    float acc = warp_sum(ok ? dot_row<NX>(w, xr) : 0.f);
                    if (lane == 0 && CHKS(cx.red + out_i * g.sw + ks, 4, 46))
                        cx.red[out_i * g.sw + ks] = acc;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&cx.empty[pg]);
    }
}

// Stages an input vector of n floats into xbuf (coalesced, from L2), with
// optional RMSNorm (x / sqrt(mean(x^2) + eps) * gain). src_bf16 selects a
// bf16 source row (the embedding of the current token).
__device__ void stage_input(const Params &p, const Ctx &cx, const float *src,
                            const uint16_t *src_bf16, int n, const uint16_t *gain) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float ss = 0.f;
    for (int i = tid * 4; i < n; i += kConsumerThreads * 4) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (src_bf16) {
            if (CHK(src_bf16 + i, 8, 9)) {
                uint2 b = __ldg(reinterpret_cast<const uint2 *>(src_bf16 + i));
                v = make_float4(bf_lo(b.x), bf_hi(b.x), bf_lo(b.y), bf_hi(b.y));
            }
        } else if (CHK(src + i, 16, 10)) {
            v = __ldcg(reinterpret_cast<const float4 *>(src + i));
        }
        if (CHKS(cx.xbuf + i, 16, 47)) *reinterpret_cast<float4 *>(cx.xbuf + i) = v;
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    if (!gain) {
        consumer_sync();
        return;
    }
    ss = warp_sum(ss);
    if (lane == 0) cx.misc->red8[warp] = ss;
    consumer_sync();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) tot += cx.misc->red8[w];
    const float rstd = 1.0f / sqrtf(tot / (float)n + p.eps);
    for (int i = tid; i < n; i += kConsumerThreads)
        if (CHK(gain + i, 2, 11)) cx.xbuf[i] = cx.xbuf[i] * rstd * bf16f(__ldg(gain + i));
    consumer_sync();
}

__device__ __forceinline__ int current_token(const Params &p) {
    if (p.d_token && !CHK(p.d_token, 4, 33)) return -1;
    return p.d_token ? *(volatile const int32_t *)p.d_token : p.token;
}

template <int NX>
__device__ void gemv_dispatch_nx(const Params &p, const Ctx &cx, const Instr &in, const Geo &g,
                                 const float *xsrc, bool xglobal, uint32_t &t, bool &bad) {
    gemv_tiles<NX>(p, cx, in, g, xsrc, xglobal, t, bad);
}

__device__ void run_gemv_tiles(const Params &p, const Ctx &cx, const Instr &in, const Geo &g,
                               const float *xsrc, bool xglobal, uint32_t &t, bool &bad) {
    switch (g.nx) {
        case 8: gemv_dispatch_nx<8>(p, cx, in, g, xsrc, xglobal, t, bad); break;
        case 16: gemv_dispatch_nx<16>(p, cx, in, g, xsrc, xglobal, t, bad); break;
        case 24: gemv_dispatch_nx<24>(p, cx, in, g, xsrc, xglobal, t, bad); break;
        case 32: gemv_dispatch_nx<32>(p, cx, in, g, xsrc, xglobal, t, bad); break;
        case 40: gemv_dispatch_nx<40>(p, cx, in, g, xsrc, xglobal, t, bad); break;
        case 48: gemv_dispatch_nx<48>(p, cx, in, g, xsrc, xglobal, t, bad); break;
        case 56: gemv_dispatch_nx<56>(p, cx, in, g, xsrc, xglobal, t, bad); break;
        default: gemv_dispatch_nx<64>(p, cx, in, g, xsrc, xglobal, t, bad); break;
    }
}

__device__ void do_gemv(const Params &p, const Ctx &cx, const Instr &in, uint32_t &t, bool &bad) {
    const Geo &g = geo_of(p, in.op);
    const int tid = threadIdx.x;
    const int l = in.layer;
    const LayerW *lw = p.layers + l;
    // ---- prologue: the input vector
    const float *xsrc = cx.xbuf;
    bool xglobal = false;
    switch (in.op) {
        case OP_QKV: {
            const int tok = current_token(p);
            if (l == 0)
                stage_input(p, cx, nullptr, p.embed + (size_t)tok * p.d, p.d, lw->attn_norm);
            else
                stage_input(p, cx, p.x, nullptr, p.d, lw->attn_norm);
            break;
        }
        case OP_GATEUP: stage_input(p, cx, p.x, nullptr, p.d, lw->mlp_norm); break;
        case OP_LMHEAD: stage_input(p, cx, p.x, nullptr, p.d, p.final_norm); break;
        case OP_OPROJ: stage_input(p, cx, p.att + (size_t)l * p.Hq * p.hd, nullptr, p.Hq * p.hd, nullptr); break;
        default:  // OP_DOWN: K = F may exceed the staging buffer; slices come from L2
            xsrc = p.h + (size_t)l * p.F;
            xglobal = true;
            break;
    }
    // ---- tiles
    run_gemv_tiles(p, cx, in, g, xsrc, xglobal, t, bad);
    bad = consumer_sync_any(bad);
    if (bad) return;
    // ---- epilogue: combine K-slices, apply the op's output transform
    const int n = in.a1, r0 = in.a0, sw = g.sw;
    switch (in.op) {
        case OP_QKV: {
            float *dst = p.qkv + (size_t)l * (p.Hq + 2 * p.Hkv) * p.hd +
                         (in.mat == 0 ? 0 : (in.mat == 1 ? p.Hq * p.hd : (p.Hq + p.Hkv) * p.hd)) + r0;
            for (int i = tid; i < n; i += kConsumerThreads) {
                float v = 0.f;
                for (int s = 0; s < sw; ++s) v += cx.red[i * sw + s];
                if (CHK(dst + i, 4, 12)) dst[i] = v;
            }
            break;
        }
        case OP_OPROJ: {
            const int tok = current_token(p);
            for (int i = tid; i < n; i += kConsumerThreads) {
                float v = 0.f;
                for (int s = 0; s < sw; ++s) v += cx.red[i * sw + s];
                float res = 0.f;
                if (l == 0) {
                    if (CHK(p.embed + (size_t)tok * p.d + r0 + i, 2, 13))
                        res = bf16f(__ldg(p.embed + (size_t)tok * p.d + r0 + i));
                } else if (CHK(p.x + r0 + i, 4, 14)) {
                    res = ldcg(p.x + r0 + i);
                }
                if (CHK(p.x + r0 + i, 4, 15)) p.x[r0 + i] = res + v;
            }
            break;
        }
        case OP_GATEUP: {
            float *dst = p.h + (size_t)l * p.F + r0;
            for (int i = tid; i < n; i += kConsumerThreads) {
                float gv = 0.f, uv = 0.f;
                for (int s = 0; s < sw; ++s) {
                    gv += cx.red[i * sw + s];
                    uv += cx.red[(n + i) * sw + s];
                }
                if (CHK(dst + i, 4, 16)) dst[i] = gv / (1.0f + expf(-gv)) * uv;
            }
            break;
        }
        case OP_DOWN: {
            for (int i = tid; i < n; i += kConsumerThreads) {
                float v = 0.f;
                for (int s = 0; s < sw; ++s) v += cx.red[i * sw + s];
                if (CHK(p.x + r0 + i, 4, 17)) p.x[r0 + i] = ldcg(p.x + r0 + i) + v;
            }
            break;
        }
        default: {  // OP_LMHEAD
            unsigned long long best = 0ull;
            for (int i = tid; i < n; i += kConsumerThreads) {
                float v = 0.f;
                for (int s = 0; s < sw; ++s) v += cx.red[i * sw + s];
                if (p.out_logits && CHK(p.out_logits + r0 + i, 4, 18)) p.out_logits[r0 + i] = v;
                const unsigned long long k = argmax_key(v, (uint32_t)(r0 + i));
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
                __threadfence();
                const uint32_t old = CHK(p.ctr + p.cl.lm_arrive, 4, 31)
                                         ? atom_acq_rel_add(p.ctr + p.cl.lm_arrive, 1u) : 0u;
                if (old == (uint32_t)p.n_lm - 1u) {
                    unsigned long long g2 = 0ull;
                    for (int s = 0; s < p.n_lm; ++s) {
                        const unsigned long long v = CHK(p.lm_part + s, 8, 20) ? __ldcg(p.lm_part + s) : 0ull;
                        g2 = v > g2 ? v : g2;
                    }
                    if (CHK(p.out_token, 4, 21))
                        *p.out_token = (int32_t)(0xFFFFFFFFu - (uint32_t)(g2 & 0xFFFFFFFFull));
                }
            }
            break;
        }
    }
}

// ---------------------------------------------------------------------------
// Attention: one KV split of one kv head (all G query heads of its group).
// Scores in log2 units (q pre-scaled by log2(e)/sqrt(hd)); each warp keeps an
// online-softmax state over its positions; warps are merged in shared
// memory, splits are merged by the last split to arrive (log-sum-exp merge).
// ---------------------------------------------------------------------------
template <int HD>
struct AttnWarpState {
    static constexpr int DPL = HD / 32;  // output dims per lane
    float m[kMaxG], l[kMaxG], o[kMaxG][DPL];
};

// One chunk of up to PPW positions for this warp. Kp/Vp point at the first
// position's key/value row (bf16, HD each); npos valid positions.
template <int HD>
__device__ __forceinline__ void attn_chunk(AttnWarpState<HD> &st, const uint16_t *Kp,
                                           const uint16_t *Vp, int npos, const float *q, int G,
                                           float *pbuf) {
    constexpr int PPW = (HD == 64) ? 16 : 8;  // positions per warp per chunk
    constexpr int DPL = HD / 32;
    const int lane = threadIdx.x & 31;
    const int pj = lane % PPW, part = lane / PPW;
    const bool valid = pj < npos;
    float s[kMaxG];
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) s[g] = 0.f;
    if (valid) {
        const uint4 *kr = reinterpret_cast<const uint4 *>(Kp + (size_t)pj * HD + part * 32);
        uint4 kw[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) kw[c] = kr[c];
#pragma unroll
        for (int g = 0; g < kMaxG; ++g) {
            if (g < G) {
                const float4 *qg = reinterpret_cast<const float4 *>(q + g * HD + part * 32);
                float a = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float4 q0 = qg[2 * c], q1 = qg[2 * c + 1];
                    a = fmaf(bf_lo(kw[c].x), q0.x, a);
                    a = fmaf(bf_hi(kw[c].x), q0.y, a);
                    a = fmaf(bf_lo(kw[c].y), q0.z, a);
                    a = fmaf(bf_hi(kw[c].y), q0.w, a);
                    a = fmaf(bf_lo(kw[c].z), q1.x, a);
                    a = fmaf(bf_hi(kw[c].z), q1.y, a);
                    a = fmaf(bf_lo(kw[c].w), q1.z, a);
                    a = fmaf(bf_hi(kw[c].w), q1.w, a);
                }
                s[g] = a;
            }
        }
    }
    // sum the LPP parts of each position
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) {
#pragma unroll
        for (int o = PPW; o < 32; o <<= 1) s[g] += __shfl_xor_sync(0xFFFFFFFFu, s[g], o);
    }
    float pv[kMaxG];
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) {
        if (g < G) {
            float mloc = valid ? s[g] : -INFINITY;
#pragma unroll
            for (int o = 1; o < PPW; o <<= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xFFFFFFFFu, mloc, o));
            const float mnew = fmaxf(st.m[g], mloc);
            const float corr = exp2f(st.m[g] - mnew);
            pv[g] = valid ? exp2f(s[g] - mnew) : 0.f;
            float ls = pv[g];
#pragma unroll
            for (int o = 1; o < PPW; o <<= 1) ls += __shfl_xor_sync(0xFFFFFFFFu, ls, o);
            st.l[g] = st.l[g] * corr + ls;
#pragma unroll
            for (int e = 0; e < DPL; ++e) st.o[g][e] *= corr;
            st.m[g] = mnew;
        }
    }
    if (part == 0 && valid) {
#pragma unroll
        for (int g = 0; g < kMaxG; ++g)
            if (g < G) pbuf[pj * kMaxG + g] = pv[g];
    }
    __syncwarp();
    for (int j = 0; j < npos; ++j) {
        const uint16_t *vr = Vp + (size_t)j * HD + lane * DPL;
        float v[DPL];
        if constexpr (DPL == 2) {
            const uint32_t u = *reinterpret_cast<const uint32_t *>(vr);
            v[0] = bf_lo(u);
            v[1] = bf_hi(u);
        } else {
            const uint2 u = *reinterpret_cast<const uint2 *>(vr);
            v[0] = bf_lo(u.x);
            v[1] = bf_hi(u.x);
            v[2] = bf_lo(u.y);
            v[3] = bf_hi(u.y);
        }
#pragma unroll
        for (int g = 0; g < kMaxG; ++g) {
            if (g < G) {
                const float pg = pbuf[j * kMaxG + g];
#pragma unroll
                for (int e = 0; e < DPL; ++e) st.o[g][e] = fmaf(pg, v[e], st.o[g][e]);
            }
        }
    }
    __syncwarp();
}

template <int HD>
__device__ void do_attn_hd(const Params &p, const Ctx &cx, const Instr &in, uint32_t &t, bool &bad) {
    constexpr int PPW = (HD == 64) ? 16 : 8;
    constexpr int DPL = HD / 32;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int l = in.layer, kvh = in.a0, split = in.a1, G = p.G;
    const AttnRange r = attn_range(p, split);
    const int qkv_stride = (p.Hq + 2 * p.Hkv) * p.hd;
    const float *qkv = p.qkv + (size_t)l * qkv_stride;
    // shared scratch: q [G][HD] | knew [HD] bf16 | vnew [HD] bf16 | warp states
    // [8][G][HD+2]; the host checks G*HD + HD + 8*G*(HD+2) <= kXbufFloats.
    float *qs = cx.xbuf;
    uint16_t *knew = reinterpret_cast<uint16_t *>(cx.xbuf + G * HD);
    uint16_t *vnew = knew + HD;
    float *wst = cx.xbuf + G * HD + HD;
    float *pbuf = cx.red + warp * (PPW * kMaxG);

    if (r.active) {
        if (tid == 0) cx.misc->flag = wait_counter(p, p.ctr + in.wait_ctr, (uint32_t)in.wait_target);
        consumer_sync();
        if (!cx.misc->flag) bad = true;
    }
    if (r.active && !bad) {
        // q of the group's heads, rotated and pre-scaled; the new key/value.
        const float qscale = 1.4426950408889634f / sqrtf((float)HD);
        const float *rope = p.rope + (size_t)p.pos * HD;  // [HD/2][2]
        for (int idx = tid; idx < G * (HD / 2); idx += kConsumerThreads) {
            const int g = idx / (HD / 2), i = idx % (HD / 2);
            const float *qh = qkv + (size_t)(kvh * G + g) * HD;
            if (!(CHK(qh + i, 4, 22) && CHK(qh + i + HD / 2, 4, 22) && CHK(rope + 2 * i, 8, 28) &&
                  CHKS(qs + g * HD + i + HD / 2, 4, 48)))
                continue;
            const float a = ldcg(qh + i), b = ldcg(qh + i + HD / 2);
            const float c = rope[2 * i], s = rope[2 * i + 1];
            qs[g * HD + i] = (a * c - b * s) * qscale;
            qs[g * HD + i + HD / 2] = (b * c + a * s) * qscale;
        }
        if (r.has_new) {
            const float *kh = qkv + (size_t)p.Hq * HD + (size_t)kvh * HD;
            const float *vh = qkv + (size_t)(p.Hq + p.Hkv) * HD + (size_t)kvh * HD;
            const size_t cache_off = (((size_t)l * p.max_batch) * p.Hkv + kvh) * p.max_seq * HD +
                                     (size_t)p.pos * HD;
            for (int i = tid; i < HD / 2; i += kConsumerThreads) {
                if (!(CHK(kh + i, 4, 23) && CHK(kh + i + HD / 2, 4, 23) && CHK(vh + i, 4, 23) &&
                      CHK(vh + i + HD / 2, 4, 23) && CHK(p.kc + cache_off + i, 2, 24) &&
                      CHK(p.kc + cache_off + i + HD / 2, 2, 24) && CHK(p.vc + cache_off + i, 2, 24) &&
                      CHK(p.vc + cache_off + i + HD / 2, 2, 24) && CHK(rope + 2 * i, 8, 28) &&
                      CHKS(vnew + i + HD / 2, 2, 49)))
                    continue;
                const float a = ldcg(kh + i), b = ldcg(kh + i + HD / 2);
                const float c = rope[2 * i], s = rope[2 * i + 1];
                const uint16_t k0 = f2bf(a * c - b * s), k1 = f2bf(b * c + a * s);
                const uint16_t v0 = f2bf(ldcg(vh + i)), v1 = f2bf(ldcg(vh + i + HD / 2));
                knew[i] = k0;
                knew[i + HD / 2] = k1;
                vnew[i] = v0;
                vnew[i + HD / 2] = v1;
                p.kc[cache_off + i] = k0;
                p.kc[cache_off + i + HD / 2] = k1;
                p.vc[cache_off + i] = v0;
                p.vc[cache_off + i + HD / 2] = v1;
            }
        }
        consumer_sync();
    }
    // per-warp online softmax over the split's tiles
    AttnWarpState<HD> st;
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) {
        st.m[g] = -INFINITY;
        st.l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) st.o[g][e] = 0.f;
    }
    const int nt = r.active ? (r.t1 - r.t0 + p.ppt - 1) / p.ppt : 0;
    for (int j = 0; j < nt; ++j, ++t) {
        const int pg = t % kPages;
        if (!bad && !wait_bar(p, &cx.full[pg], (t / kPages) & 1)) bad = true;
        if (!bad) {
            const int ts = r.t0 + j * p.ppt;
            int n = r.t1 - ts;
            if (n > p.ppt) n = p.ppt;
            int np = n - warp * PPW;
            np = np > PPW ? PPW : np;
            if (np > 0 && CHKS(cx.pages + (size_t)pg * kPageBytes + (size_t)(warp * PPW + np) * HD * 2 - 2, 2, 50) &&
                CHKS(pbuf + PPW * kMaxG - 1, 4, 51)) {
                const uint16_t *Kp = reinterpret_cast<const uint16_t *>(cx.pages + (size_t)pg * kPageBytes) +
                                     (size_t)warp * PPW * HD;
                const uint16_t *Vp = reinterpret_cast<const uint16_t *>(cx.pages + (size_t)pg * kPageBytes +
                                                                          kPageBytes / 2) +
                                     (size_t)warp * PPW * HD;
                attn_chunk<HD>(st, Kp, Vp, np, qs, G, pbuf);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&cx.empty[pg]);
    }
    bad = consumer_sync_any(bad);
    if (r.active && !bad) {
        if (r.has_new && warp == kConsumerWarps - 1) attn_chunk<HD>(st, knew, vnew, 1, qs, G, pbuf);
        // warp states -> shared
        float *my = wst + (size_t)warp * G * (HD + 2);
        if (!CHKS(my + G * (HD + 2) - 1, 4, 52)) my = wst;
        for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int e = 0; e < DPL; ++e) my[g * (HD + 2) + lane * DPL + e] = st.o[g][e];
            if (lane == 0) {
                my[g * (HD + 2) + HD] = st.m[g];
                my[g * (HD + 2) + HD + 1] = st.l[g];
            }
        }
        consumer_sync();
        // combine the warps into this split's partial (o unnormalised, m, l)
        float *dst = p.part + ((size_t)l * p.Hq + (size_t)kvh * G) * p.S * (HD + 2);
        for (int idx = tid; idx < G * (HD + 2); idx += kConsumerThreads) {
            const int g = idx / (HD + 2), e = idx % (HD + 2);
            float M = -INFINITY;
            for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, wst[(w * G + g) * (HD + 2) + HD]);
            float acc = 0.f;
            if (e == HD) {
                acc = M;
            } else if (M != -INFINITY) {
                const int src = (e == HD + 1) ? HD + 1 : e;
                for (int w = 0; w < kConsumerWarps; ++w) {
                    const float mw = wst[(w * G + g) * (HD + 2) + HD];
                    if (mw != -INFINITY) acc += wst[(w * G + g) * (HD + 2) + src] * exp2f(mw - M);
                }
            }
            if (CHK(dst + ((size_t)g * p.S + split) * (HD + 2) + e, 4, 25))
                dst[((size_t)g * p.S + split) * (HD + 2) + e] = acc;
        }
    }
    consumer_sync();
    // arrival; the last split of this kv head merges all active splits
    if (tid == 0) {
        __threadfence();
        const uint32_t old = CHK(p.ctr + p.cl.merge + l * p.Hkv + kvh, 4, 31)
                                 ? atom_acq_rel_add(p.ctr + p.cl.merge + l * p.Hkv + kvh, 1u) : 0u;
        cx.misc->flag = (old == (uint32_t)p.S - 1u);
    }
    consumer_sync();
    if (cx.misc->flag && !bad) {
        const int seff = attn_seff(p);
        const float *src = p.part + ((size_t)l * p.Hq + (size_t)kvh * G) * p.S * (HD + 2);
        float *out = p.att + (size_t)l * p.Hq * HD + (size_t)kvh * G * HD;
        for (int idx = tid; idx < G * HD; idx += kConsumerThreads) {
            const int g = idx / HD, e = idx % HD;
            const float *sg = src + (size_t)g * p.S * (HD + 2);
            if (!(CHK(sg, 4, 26) && CHK(sg + (size_t)seff * (HD + 2) - 1, 4, 26) && CHK(out + idx, 4, 27)))
                continue;
            float M = -INFINITY;
            for (int s = 0; s < seff; ++s) M = fmaxf(M, ldcg(sg + (size_t)s * (HD + 2) + HD));
            float num = 0.f, den = 0.f;
            for (int s = 0; s < seff; ++s) {
                const float ms = ldcg(sg + (size_t)s * (HD + 2) + HD);
                if (ms == -INFINITY) continue;
                const float wgt = exp2f(ms - M);
                num += ldcg(sg + (size_t)s * (HD + 2) + e) * wgt;
                den += ldcg(sg + (size_t)s * (HD + 2) + HD + 1) * wgt;
            }
            out[idx] = num / den;
        }
        consumer_sync();
        if (tid == 0) {
            __threadfence();
            if (CHK(p.ctr + p.cl.attn_done + l, 4, 30)) red_release_add(p.ctr + p.cl.attn_done + l, 1u);
        }
    }
}

__device__ void do_attn(const Params &p, const Ctx &cx, const Instr &in, uint32_t &t, bool &bad) {
    if (p.hd == 64)
        do_attn_hd<64>(p, cx, in, t, bad);
    else
        do_attn_hd<128>(p, cx, in, t, bad);
}

// ---------------------------------------------------------------------------
// Consumer: interprets the queue.
// ---------------------------------------------------------------------------
__device__ void consumer(const Params &p, const Ctx &cx, int qb, int qe) {
    const int tid = threadIdx.x;
    uint32_t t = 0;
    bool bad = false;
    long long *trace = p.trace ? p.trace + (size_t)blockIdx.x * p.trace_cap * 5 : nullptr;
    for (int i = qb; i < qe && !bad; ++i) {
        const Instr in = load_instr(p, i);
        const uint64_t tw = trace ? gtimer() : 0;
        if (in.op != OP_ATTN && in.wait_ctr >= 0) {
            if (tid == 0) cx.misc->flag = wait_counter(p, p.ctr + in.wait_ctr, (uint32_t)in.wait_target);
            consumer_sync();
            if (!cx.misc->flag) {
                bad = true;
                break;
            }
        }
        const uint64_t ts = trace ? gtimer() : 0;
        if (in.op == OP_ATTN)
            do_attn(p, cx, in, t, bad);
        else
            do_gemv(p, cx, in, t, bad);
        consumer_sync();
        if (bad) break;
        if (tid == 0) {
            if (in.sig_n > 0) {
                __threadfence();
                for (int c = 0; c < in.sig_n; ++c)
                    if (CHK(p.ctr + in.sig_ctr + c, 4, 30)) red_release_add(p.ctr + in.sig_ctr + c, 1u);
            }
            if (trace && (i - qb) < p.trace_cap && CHK(trace + (size_t)(i - qb) * 5, 40, 34)) {
                long long *rec = trace + (size_t)(i - qb) * 5;
                rec[0] = blockIdx.x;
                rec[1] = in.op;
                rec[2] = (long long)tw;
                rec[3] = (long long)ts;
                rec[4] = (long long)gtimer();
            }
        }
    }
    if (bad && tid == 0) cx.misc->aborted = 1;
}

__global__ void __launch_bounds__(kThreads, 1) mk_megakernel(const Params prm) {
    uint8_t *smem = mk_smem;
    // Launch parameters are copied to shared memory once; every device
    // function reads them from there (no generic pointer into param space).
    Params *sp = reinterpret_cast<Params *>(smem + kSmemParams);
    Ctx cx;
    cx.pages = smem + kSmemPages;
    cx.xbuf = reinterpret_cast<float *>(smem + kSmemXbuf);
    cx.red = reinterpret_cast<float *>(smem + kSmemRed);
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
        cx.misc->aborted = 0;
        cx.misc->n_issued = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    const Params &p = *sp;
    const int *qrow = p.q_begin + (size_t)blockIdx.x * (p.n_stages + 1);
    bool run = CHK(qrow + p.stage_lo, 4, 2) && CHK(qrow + p.stage_hi, 4, 2) &&
               CHK(p.status, 4, 32) && CHK(p.abort_flag, 4, 32) && CHK(p.exit_ctr, 4, 32);
    const int qb = run ? __ldg(qrow + p.stage_lo) : 0, qe = run ? __ldg(qrow + p.stage_hi) : 0;
    run = run && *(volatile int32_t *)p.status == DS_OK;
    if (run) {
        const int tok = current_token(p);
        if (tok < 0 || tok >= p.V) {
            if (tid == 0) {
                atomicCAS(p.status, DS_OK, DS_BAD_TOKEN);
                atomicExch(p.abort_flag, 1);
            }
            run = false;
        }
    }
    if (run) {
        if (warp == kConsumerWarps) {
            if (lane == 0) producer(p, cx, qb, qe);
        } else {
            consumer(p, cx, qb, qe);
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
    // End of step: the last CTA out resets the counters for the next step.
    if (p.reset_at_exit && tid == 0 && CHK(p.exit_ctr, 4, 32) &&
        CHK(p.ctr + p.cl.total - 1, 4, 32)) {
        __threadfence();
        const uint32_t old = atomicAdd(p.exit_ctr, 1u);
        if (old == gridDim.x - 1) {
            for (int c = 0; c < p.cl.total; ++c) p.ctr[c] = 0u;
            *p.abort_flag = 0;
            *p.exit_ctr = 0u;
            __threadfence();
        }
    }
}

}  // namespace mk

// ---------------------------------------------------------------------------
// Host-side launch helpers (called from mk_host.cpp)
// ---------------------------------------------------------------------------
extern "C" cudaError_t mk_kernel_configure(void) {
    return cudaFuncSetAttribute(mk::mk_megakernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                mk::kSmemBytes);
}

extern "C" cudaError_t mk_kernel_launch(const mk::Params *p, int n_sm, int cooperative,
                                        cudaStream_t stream) {
    if (cooperative) {
        void *args[] = {const_cast<mk::Params *>(p)};
        return cudaLaunchCooperativeKernel((const void *)mk::mk_megakernel, dim3(n_sm),
                                           dim3(mk::kThreads), args, mk::kSmemBytes, stream);
    }
    mk::mk_megakernel<<<n_sm, mk::kThreads, mk::kSmemBytes, stream>>>(*p);
    return cudaGetLastError();
}

extern "C" cudaError_t mk_kernel_occupancy(int *blocks_per_sm) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, mk::mk_megakernel,
                                                         mk::kThreads, mk::kSmemBytes);
}
