// mk_host.cpp — host scheduler and C ABI of the decode megakernel.
//
// The scheduler plans, once per model, one instruction sequence per SM and a
// dependency count for every instruction ("Revolution der
// KI-Beschleunigung: Wie ein Low-Latency Megakernel den Llama-1B Turbo
// zündet", dasgeld.co: sequences pre-planned on the host and reused for many
// forward passes without recompiling; counters in global memory that tell
// an instruction when its inputs are ready). The plan is uploaded in
// mk_create and every decode step is then one launch of the interpreter.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <numeric>
#include <string>
#include <vector>

#include "../../include/mk.h"
#include "mk_plan.h"
#include "mk_prefill.h"

extern "C" cudaError_t mk_kernel_configure(void);
extern "C" cudaError_t mk_kernel_launch(const mk::Params *p, int n_sm, int cooperative,
                                        cudaStream_t stream);
extern "C" cudaError_t mk_kernel_occupancy(int *blocks_per_sm);
extern "C" cudaError_t mk_convert_bf16_f16(const void *src, void *dst, size_t n, unsigned long long *out_of_range,
                                           cudaStream_t stream);
extern "C" size_t mk_filter_lists_keys(int B, int V);
extern "C" cudaError_t mk_filtered_draw_batch(const float *logits, int B, int V, int K, float top_p, float inv_temp,
                                              const int32_t *positions, int pos0, int slot0, uint64_t seed,
                                              unsigned long long *lists, int32_t *out_tokens, cudaStream_t stream);
extern "C" cudaError_t mk_sampled_draw_batch(const float *logits, int B, int V, float inv_temp,
                                             const int32_t *positions, int pos0, uint64_t seed,
                                             unsigned long long *keys, int32_t *out_tokens, cudaStream_t stream);
extern "C" cudaError_t mk_batch_final_norm(const float *x, int B, int d, const uint16_t *gain, float eps, uint16_t *hi,
                                           uint16_t *lo, cudaStream_t stream);
extern "C" cudaError_t mk_noise_launch(int n, int pos, int slot, uint64_t seed, const uint32_t *words,
                                       uint32_t *out_words, float *out_noise, cudaStream_t stream);

namespace {

thread_local std::string g_err;

int fail(int code, const std::string &msg) {
    g_err = msg;
    return code;
}

int cuda_fail(cudaError_t e, const char *what) {
    return fail(e == cudaErrorMemoryAllocation ? MK_ERR_NOMEM : MK_ERR_CUDA,
                std::string(what) + ": " + cudaGetErrorString(e));
}

using mk::Geo;
using mk::Instr;

// ---------------------------------------------------------------------------
// Tile geometry for an input length K (see Geo in mk_plan.h).
// ---------------------------------------------------------------------------
bool make_geo(int K, Geo &g, int max_nx = 32) {
    if (K <= 0 || K % 256 != 0 || K > 16384) return false;
    int sw = 1;
    while (K / sw > 32 * max_nx || (K / sw) % 256 != 0) {
        sw *= 2;
        if (sw > mk::kConsumerWarps) return false;
    }
    g.K = K;
    g.sw = sw;
    g.rw = mk::kConsumerWarps / sw;
    g.kslice = K / sw;
    g.nx = g.kslice / 32;
    const int row_bytes = K * 2;
    g.m = mk::kPageBytes / (g.rw * row_bytes);
    if (g.m < 1) return false;
    g.rt = g.rw * g.m;
    g.pad = 0;
    return true;
}

// Batched steps: tiles of rt rows x a K-chunk of KC = min(K, 2048) columns,
// 8 rows and a 256-wide slice per warp (see mk_plan.h).
bool make_geo_batch(int K, Geo &g) {
    // K-chunks of KC <= 1024 columns, 128 per warp; 16 rows per warp
    const int KC = std::min(K, 1024);
    if (K <= 0 || K % KC != 0 || (KC != 128 && KC != 256 && KC != 512 && KC != 1024)) return false;
    g.K = K;
    g.sw = KC / 128;
    g.rw = mk::kConsumerWarps / g.sw;
    g.m = 16;
    g.rt = g.rw * g.m;
    g.nx = 4;
    g.kslice = 128;
    g.pad = KC;
    return g.rt * KC * 2 <= mk::kPageBytes;
}

struct Plan {
    int nb = 1;  // sequences of one step
    int n_sm = 0, S = 1, ppt = 0, n_lm = 0, n_stages = 0;
    int attn_parts = 1;  // instructions sharing one (kv head, split): its query heads split between them
    mk::CtrLayout cl{};
    Geo geo_qkv{}, geo_o{}, geo_gu{}, geo_down{}, geo_lm{};
    std::vector<std::vector<Instr>> q;
    size_t n_instr() const {
        size_t n = 0;
        for (auto &v : q) n += v.size();
        return n;
    }
};

int check_config(const mk_config *c) {
    if (!c) return fail(MK_ERR_INVALID_ARG, "config is NULL");
    if (c->n_layers < 1 || c->n_layers > 4096 || c->d_model < 1 || c->n_heads < 1 ||
        c->n_kv_heads < 1 || c->head_dim < 1 || c->ffn_dim < 1 || c->vocab < 1 || c->max_seq < 1 ||
        c->max_batch < 1 || c->attn_splits < 0)
        return fail(MK_ERR_INVALID_ARG, "config has a non-positive size");
    if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f))
        return fail(MK_ERR_INVALID_ARG, "rms_eps must be >= 0 and rope_theta > 0");
    if (c->head_dim != 64 && c->head_dim != 128)
        return fail(MK_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (c->n_heads % c->n_kv_heads != 0)
        return fail(MK_ERR_INVALID_ARG, "n_heads must be a multiple of n_kv_heads");
    const int G = c->n_heads / c->n_kv_heads, hd = c->head_dim;
    if (G > 4 || G * (hd / 16 * 20) + hd + mk::kConsumerWarps * G * (hd + 4) > mk::kXbufFloats)
        return fail(MK_ERR_UNSUPPORTED, "too many query heads per kv head for the attention scratch");
    const int qd = c->n_heads * hd;
    if (c->d_model % 256 || qd % 256 || c->ffn_dim % 256)
        return fail(MK_ERR_UNSUPPORTED, "d_model, n_heads*head_dim and ffn_dim must be multiples of 256");
    if (c->d_model > mk::kMaxStaged || qd > mk::kMaxStaged)
        return fail(MK_ERR_UNSUPPORTED, "d_model and n_heads*head_dim must be <= 4096");
    if (c->n_layers > 127) return fail(MK_ERR_UNSUPPORTED, "at most 127 layers (activation tag versions)");
    if (c->ffn_dim > mk::kMaxStagedLong) return fail(MK_ERR_UNSUPPORTED, "ffn_dim must be <= 8192");
    const double kv_elems = (double)c->n_layers * c->max_batch * c->n_kv_heads * c->max_seq * hd;
    if (kv_elems * 2 > 9.0e18) return fail(MK_ERR_INVALID_ARG, "KV cache too large");
    return MK_OK;
}

// Balanced contiguous split of N rows of one stage across the SMs. The
// N % n_sm extra rows go to the SMs with the least bytes so far, so the
// per-SM byte totals over the whole step stay even.
struct Chunk {
    int sm, r0, n;
};

std::vector<Chunk> split_rows(int N, double cost_per_row, std::vector<double> &load, int max_rows,
                              const std::vector<char> *excluded = nullptr) {
    const int n_sm = (int)load.size();
    std::vector<int> order;
    for (int sm = 0; sm < n_sm; ++sm)
        if (!excluded || !(*excluded)[sm]) order.push_back(sm);
    const int n_use = (int)order.size();
    const int base = N / n_use, extra = N % n_use;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return load[a] < load[b]; });
    std::vector<int> cnt(n_sm, 0);
    for (int i = 0; i < n_use; ++i) cnt[order[i]] = base + (i < extra ? 1 : 0);
    std::vector<Chunk> out;
    int r = 0;
    for (int sm = 0; sm < n_sm; ++sm) {
        int left = cnt[sm];
        load[sm] += left * cost_per_row;
        while (left > 0) {
            const int n = std::min(left, max_rows);
            out.push_back({sm, r, n});
            r += n;
            left -= n;
        }
    }
    return out;
}

int build_plan(const mk_config *c, int n_sm, Plan &P, int nb) {
    int rc = check_config(c);
    if (rc) return rc;
    if (n_sm < 1 || n_sm > 4096) return fail(MK_ERR_INVALID_ARG, "bad SM count");
    const int L = c->n_layers, d = c->d_model, Hq = c->n_heads, Hkv = c->n_kv_heads,
              hd = c->head_dim, F = c->ffn_dim, V = c->vocab, G = Hq / Hkv;
    const int qd = Hq * hd, kvd = Hkv * hd;
    P = Plan();
    P.n_sm = n_sm;
    P.nb = nb;
    if (nb > 1) {
        // batched steps: hd 64 instances
        // (the LM head of a batched step runs after the launch, on the tensor
        // cores: no LM-head instructions in this plan)
        if (nb > mk::kMaxBatch || hd != 64 || !make_geo_batch(d, P.geo_qkv) ||
            !make_geo_batch(qd, P.geo_o) || !make_geo_batch(d, P.geo_gu) || !make_geo_batch(F, P.geo_down))
            return fail(MK_ERR_UNSUPPORTED, "no batched tile geometry for this model");
    } else {
        // input floats per lane: 32 gives the fewest K-slices per row
        auto geo = [&](int K, Geo &g) { return make_geo(K, g, 32); };
        if (!geo(d, P.geo_qkv) || !geo(qd, P.geo_o) || !geo(d, P.geo_gu) || !geo(F, P.geo_down) ||
            !geo(d, P.geo_lm))
            return fail(MK_ERR_UNSUPPORTED, "no tile geometry for these input lengths");
    }
    if (P.geo_gu.rt < 2 || P.geo_gu.rt % 2)
        return fail(MK_ERR_UNSUPPORTED, "gate/up tile needs an even row count");
    P.ppt = (mk::kPageBytes / 2) / (hd * 2);
    const int max_tiles = (c->max_seq + P.ppt * mk::kMinSplitTiles - 1) / (P.ppt * mk::kMinSplitTiles);
    int S = std::max(1, std::min(n_sm / Hkv, max_tiles));
    if (c->attn_splits > 0) S = std::min(c->attn_splits, std::max(1, max_tiles));
    P.S = S;
    P.n_stages = mk::kStagesPerLayer * L + 1;
    auto &cl = P.cl;
    cl.qkv_grp = 0;
    cl.merge = cl.qkv_grp + L * Hkv;
    cl.attn_done = cl.merge + L * Hkv;
    cl.oproj_done = cl.attn_done + L;
    cl.gateup_done = cl.oproj_done + L;
    cl.down_done = cl.gateup_done + L;
    cl.lm_arrive = cl.down_done + L;
    cl.total = cl.lm_arrive + 1;

    P.q.assign(n_sm, {});
    std::vector<double> load(n_sm, 0.0);
    auto mk_instr = [](int op, int layer, int stage) {
        Instr in;
        std::memset(&in, 0, sizeof in);
        in.op = op;
        in.layer = layer;
        in.stage = stage;
        in.wait_ctr = -1;
        return in;
    };
    auto set_bytes = [](Instr &in, long long b) {
        in.bytes_lo = (int32_t)(b & 0xFFFFFFFFll);
        in.bytes_hi = (int32_t)(b >> 32);
    };
    // rows per instruction: what the per-row partials (batched: the shared
    // accumulators and the residual rows of every sequence) can hold
    const int cap_qkv = nb > 1 ? mk::kRedCap / mk::kMaxBatch : mk::kRedCap / P.geo_qkv.sw,
              cap_o = nb > 1 ? std::min(mk::kRedCap / mk::kMaxBatch, mk::kResidFloats / nb)
                             : std::min(mk::kRedCap / P.geo_o.sw, mk::kResidFloats),
              cap_gu = nb > 1 ? mk::kRedCap / (2 * mk::kMaxBatch) : mk::kRedCap / (2 * P.geo_gu.sw),
              cap_down = nb > 1 ? std::min(mk::kRedCap / mk::kMaxBatch, mk::kResidFloats / nb)
                                : std::min(mk::kDredFloats / P.geo_down.sw, mk::kResidFloats),
              cap_lm = nb > 1 ? 1 << 20 : mk::kRedCap / P.geo_lm.sw;
    // Short contexts: the attention of a layer runs on SMs that get no QKV
    // rows, so it starts as soon as q/k/v are published and its cached
    // keys/values are prefetched at the start of the layer. Long contexts
    // spread attention (and its KV streaming) over every SM instead.
    // A single sequence whose attention fits few SMs splits each kv head's
    // query heads over two instructions (two SMs): the attention sits on the
    // critical path between QKV and O-proj, and its time grows with the heads
    // one SM scores; both read the kv head's keys and values, one appends.
    P.attn_parts = (nb == 1 && G % 2 == 0 && Hkv * S * 2 * 4 <= n_sm) ? 2 : 1;
    const int AP = P.attn_parts;
    const double attn_cost = (2.0 * 2.0 * hd * std::ceil((double)c->max_seq / S) + 4096.0) / AP;
    const bool dedicated_attn = Hkv * S * nb * AP * 4 <= n_sm;
    int prev_down = 0;
    for (int l = 0; l < L; ++l) {
        const int st = mk::kStagesPerLayer * l;
        // ---- attention SMs of this layer (least loaded first)
        std::vector<int> attn_sm;
        std::vector<char> excluded(n_sm, 0);
        if (dedicated_attn) {
            std::vector<int> order(n_sm);
            std::iota(order.begin(), order.end(), 0);
            std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return load[a] < load[b]; });
            for (int i = 0; i < Hkv * S * nb * AP; ++i) {
                attn_sm.push_back(order[i]);
                excluded[order[i]] = 1;
            }
        }
        // ---- QKV: rows of the stacked [Wq; Wk; Wv] (an instruction may span
        // two of the matrices; its tiles are copied from both)
        std::vector<int> touch(Hkv, 0);
        auto group_of = [&](int row) {  // kv group whose attention reads stacked row `row`
            if (row < qd) return (row / hd) / G;
            if (row < qd + kvd) return (row - qd) / hd;
            return (row - qd - kvd) / hd;
        };
        for (const Chunk &ch : split_rows(qd + 2 * kvd, 2.0 * d, load, cap_qkv,
                                          dedicated_attn ? &excluded : nullptr)) {
            Instr in = mk_instr(mk::OP_QKV, l, st);
            in.mat = 0;
            in.a0 = ch.r0;
            in.a1 = ch.n;
            std::vector<char> hit(Hkv, 0);
            for (int r = ch.r0; r < ch.r0 + ch.n; ++r) hit[group_of(r)] = 1;
            int g0 = Hkv, g1 = -1;
            for (int g = 0; g < Hkv; ++g)
                if (hit[g]) {
                    g0 = std::min(g0, g);
                    g1 = std::max(g1, g);
                }
            // signal every group in [g0, g1] (a span crossing matrices may cover extra groups)
            in.sig_ctr = cl.qkv_grp + l * Hkv + g0;
            in.sig_n = g1 - g0 + 1;
            for (int g = g0; g <= g1; ++g) touch[g] += 1;
            if (l > 0) {
                in.wait_ctr = cl.down_done + (l - 1);
                in.wait_target = prev_down;
            }
            set_bytes(in, 2ll * in.a1 * d);
            P.q[ch.sm].push_back(in);
        }
        // ---- attention: Hkv x S splits (x nb sequences; `mat` = sequence; x AP
        // parts of the query heads, `slot` = part)
        for (int b = 0; b < nb; ++b)
        for (int h = 0; h < Hkv; ++h)
            for (int s = 0; s < S; ++s)
            for (int a = 0; a < AP; ++a) {
                int sm = dedicated_attn ? attn_sm[((b * Hkv + h) * S + s) * AP + a]
                                        : (int)(std::min_element(load.begin(), load.end()) - load.begin());
                load[sm] += attn_cost;
                Instr in = mk_instr(mk::OP_ATTN, l, st + 1);
                in.a0 = h;
                in.a1 = s;
                in.mat = b;
                in.slot = a;
                in.wait_ctr = cl.qkv_grp + l * Hkv + h;
                in.wait_target = touch[h];
                P.q[sm].push_back(in);
            }
        // ---- O-projection + residual
        int n_o = 0;
        for (const Chunk &ch : split_rows(d, 2.0 * qd, load, cap_o)) {
            Instr in = mk_instr(mk::OP_OPROJ, l, st + 2);
            in.a0 = ch.r0;
            in.a1 = ch.n;
            in.wait_ctr = cl.attn_done + l;
            in.wait_target = Hkv * nb;  // the last split of every (sequence, kv head)
            in.sig_ctr = cl.oproj_done + l;
            in.sig_n = 1;
            set_bytes(in, 2ll * ch.n * qd);
            P.q[ch.sm].push_back(in);
            ++n_o;
        }
        // ---- gate/up + SiLU
        int n_gu = 0;
        for (const Chunk &ch : split_rows(F, 4.0 * d, load, cap_gu)) {
            Instr in = mk_instr(mk::OP_GATEUP, l, st + 3);
            in.a0 = ch.r0;
            in.a1 = ch.n;
            in.wait_ctr = cl.oproj_done + l;
            in.wait_target = n_o;
            in.sig_ctr = cl.gateup_done + l;
            in.sig_n = 1;
            set_bytes(in, 4ll * ch.n * d);
            P.q[ch.sm].push_back(in);
            ++n_gu;
        }
        // ---- down + residual
        int n_down = 0;
        for (const Chunk &ch : split_rows(d, 2.0 * F, load, cap_down)) {
            Instr in = mk_instr(mk::OP_DOWN, l, st + 4);
            in.a0 = ch.r0;
            in.a1 = ch.n;
            in.wait_ctr = cl.gateup_done + l;
            in.wait_target = n_gu;
            in.sig_ctr = cl.down_done + l;
            in.sig_n = 1;
            set_bytes(in, 2ll * ch.n * F);
            P.q[ch.sm].push_back(in);
            ++n_down;
        }
        prev_down = n_down;
    }
    // ---- final norm + tied LM head + argmax (single-sequence steps; a batched
    // step's LM head follows its launch)
    int slot = 0;
    if (nb == 1) {
        for (const Chunk &ch : split_rows(V, 2.0 * d, load, cap_lm)) {
            Instr in = mk_instr(mk::OP_LMHEAD, L, mk::kStagesPerLayer * L);
            in.layer = 0;
            in.a0 = ch.r0;
            in.a1 = ch.n;
            in.wait_ctr = cl.down_done + (L - 1);
            in.wait_target = prev_down;
            in.slot = slot++;
            set_bytes(in, 2ll * ch.n * d);
            P.q[ch.sm].push_back(in);
        }
    }
    P.n_lm = slot;
    return MK_OK;
}

// ---------------------------------------------------------------------------
// Device image of a plan: where every buffer lives in one scratch region and
// the host arrays uploaded into it. Shared by mk_create (cudaMalloc'd region)
// and mk_decode_step_noalloc (a static device array).
// ---------------------------------------------------------------------------
struct DevBump {
    size_t off = 0;
    size_t take(size_t bytes) {
        size_t o = off;
        off += (bytes + 255) & ~size_t(255);
        return o;
    }
};

}  // namespace

#include "mk_internal.h"

namespace mkint {

struct ImageImpl {
    Plan plan;
};

int check_inputs(const mk_config *config, const mk_weights *w, const mk_kv_cache *kv) {
    int rc = check_config(config);
    if (rc) return rc;
    if (!w || !w->embed || !w->final_norm || !w->layers || !kv || !kv->k || !kv->v)
        return fail(MK_ERR_INVALID_ARG, "a weight or cache pointer is NULL");
    auto al = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    if (!al(w->embed) || !al(w->final_norm) || !al(kv->k) || !al(kv->v))
        return fail(MK_ERR_INVALID_ARG, "weights and caches must be 16-byte aligned");
    for (int l = 0; l < config->n_layers; ++l) {
        const mk_layer_weights &lw = w->layers[l];
        const void *ps[9] = {lw.attn_norm, lw.wq, lw.wk, lw.wv, lw.wo,
                             lw.mlp_norm, lw.w_gate, lw.w_up, lw.w_down};
        for (const void *q : ps) {
            if (!q) return fail(MK_ERR_INVALID_ARG, "a layer weight pointer is NULL");
            if (!al(q)) return fail(MK_ERR_INVALID_ARG, "layer weights must be 16-byte aligned");
        }
    }
    return MK_OK;
}

int check_device(int *dev, int *n_sm) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    int major = 0, minor = 0, coop = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev);
    cudaDeviceGetAttribute(n_sm, cudaDevAttrMultiProcessorCount, *dev);
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, *dev);
    if (!(major == 10 && minor == 3))
        return fail(MK_ERR_UNSUPPORTED, "built for sm_103 (GB300); this device is sm_" +
                                            std::to_string(major) + std::to_string(minor));
    if (!coop) return fail(MK_ERR_UNSUPPORTED, "device has no cooperative launch");
    e = mk_kernel_configure();
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    int bps = 0;
    e = mk_kernel_occupancy(&bps);
    if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
    if (bps < 1) return fail(MK_ERR_LAUNCH, "megakernel CTA does not fit on an SM");
    return MK_OK;
}

int make_image(const mk_config *config, const mk_weights *w, int n_sm, Image &im, int nb) {
    im = Image();
    im.impl = std::make_shared<ImageImpl>();
    Plan &P = im.impl->plan;
    int rc = build_plan(config, n_sm, P, nb);
    if (rc) return rc;
    const mk_config &c = *config;
    const int L = c.n_layers, d = c.d_model, Hq = c.n_heads, Hkv = c.n_kv_heads, hd = c.head_dim,
              F = c.ffn_dim, V = c.vocab;
    im.n_sm = P.n_sm;
    im.n_stages = P.n_stages;
    im.n_instr = P.n_instr();
    // flat queues and stage index
    im.flat.reserve(im.n_instr);
    im.qbeg.assign((size_t)P.n_sm * (P.n_stages + 1), 0);
    im.qlen.resize(P.n_sm);
    for (int s = 0; s < P.n_sm; ++s) {
        const int base = (int)im.flat.size();
        im.qlen[s] = (int)P.q[s].size();
        int k = 0;
        for (int st = 0; st <= P.n_stages; ++st) {
            while (k < (int)P.q[s].size() && P.q[s][k].stage < st) ++k;
            im.qbeg[(size_t)s * (P.n_stages + 1) + st] = base + k;
        }
        im.flat.insert(im.flat.end(), P.q[s].begin(), P.q[s].end());
    }
    // RoPE table: angle pos * theta^(-2i/hd), computed in double
    im.rope.assign((size_t)c.max_seq * hd, 0.f);
    for (int pos = 0; pos < c.max_seq; ++pos)
        for (int i = 0; i < hd / 2; ++i) {
            const double inv_freq = std::pow((double)c.rope_theta, -2.0 * i / (double)hd);
            const double a = (double)pos * inv_freq;
            im.rope[((size_t)pos * (hd / 2) + i) * 2] = (float)std::cos(a);
            im.rope[((size_t)pos * (hd / 2) + i) * 2 + 1] = (float)std::sin(a);
        }
    im.lws.resize(L);
    for (int l = 0; l < L; ++l) {
        const mk_layer_weights &lw = w->layers[l];
        im.lws[l] = {(const uint16_t *)lw.attn_norm, (const uint16_t *)lw.wq, (const uint16_t *)lw.wk,
                     (const uint16_t *)lw.wv, (const uint16_t *)lw.wo, (const uint16_t *)lw.mlp_norm,
                     (const uint16_t *)lw.w_gate, (const uint16_t *)lw.w_up, (const uint16_t *)lw.w_down};
    }
    // layout of the scratch region; [o_ctr, o_zero_end) must be zero before a step
    DevBump b;
    im.o_ctr = b.take(sizeof(uint32_t) * P.cl.total);
    im.o_exit = b.take(sizeof(uint32_t));
    im.o_status = b.take(sizeof(int32_t));
    im.o_abort = b.take(sizeof(int32_t));
    im.o_dbg = b.take(sizeof(unsigned long long) * 4);
    im.o_zero_end = b.off;
    im.o_layers = b.take(sizeof(mk::LayerW) * L);
    im.o_epoch = b.take(sizeof(uint32_t));
    // tagged words {value, tag}; x, the attention output and h hold one row
    // per sequence, or (batched steps) all kMaxBatch sequence slots interleaved
    const size_t nbv = nb > 1 ? (size_t)mk::kMaxBatch : 1;
    im.o_x = b.take(8 * nbv * d);
    im.o_qkv = b.take(8 * (size_t)L * nb * (Hq + 2 * Hkv) * hd);
    im.o_part = b.take(8 * (size_t)L * nb * Hq * P.S * (hd + 2));
    im.o_att = b.take(8 * (size_t)L * nbv * Hq * hd);
    im.o_h = b.take(8 * (size_t)L * nbv * F);
    im.o_lm = b.take(sizeof(unsigned long long) * nb * P.n_lm);
    im.o_cand = b.take(sizeof(unsigned long long) * mk::kMaxTopK * P.n_lm);
    im.o_tin = b.take(sizeof(int32_t) * nb);
    im.o_tout = b.take(sizeof(int32_t) * nb);
    im.o_logits = b.take(sizeof(float) * nb * V);
    im.o_rope = b.take(sizeof(float) * im.rope.size());
    im.o_instr = b.take(sizeof(Instr) * im.flat.size());
    im.o_qbeg = b.take(sizeof(int32_t) * im.qbeg.size());
    im.n_ranges = 6 + 9 * L;
    im.o_ranges = b.take(sizeof(unsigned long long) * 2 * im.n_ranges);
    im.total = b.off;
    return MK_OK;
}

void fill_params(const Image &im, const mk_config *config, const mk_weights *w,
                 const mk_kv_cache *kv, char *base, mk::Params &p) {
    const Plan &P = im.impl->plan;
    const mk_config &c = *config;
    p = mk::Params();
    p.L = c.n_layers; p.d = c.d_model; p.Hq = c.n_heads; p.Hkv = c.n_kv_heads; p.hd = c.head_dim;
    p.F = c.ffn_dim; p.V = c.vocab; p.max_seq = c.max_seq; p.max_batch = c.max_batch;
    p.S = P.S; p.G = c.n_heads / c.n_kv_heads; p.ppt = P.ppt; p.eps = c.rms_eps;
    p.attn_heads = p.G / P.attn_parts;
    p.n_lm = P.n_lm; p.n_stages = P.n_stages;
    p.nb = P.nb;
    p.geo_qkv = P.geo_qkv; p.geo_o = P.geo_o; p.geo_gu = P.geo_gu; p.geo_down = P.geo_down;
    p.geo_lm = P.geo_lm;
    p.cl = P.cl;
    p.embed = (const uint16_t *)w->embed;
    p.final_norm = (const uint16_t *)w->final_norm;
    p.lm_w = p.embed;
    p.layers = reinterpret_cast<const mk::LayerW *>(base + im.o_layers);
    p.kc = (uint16_t *)kv->k;
    p.vc = (uint16_t *)kv->v;
    p.xll = reinterpret_cast<uint2 *>(base + im.o_x);
    p.qkvll = reinterpret_cast<uint2 *>(base + im.o_qkv);
    p.partll = reinterpret_cast<uint2 *>(base + im.o_part);
    p.attll = reinterpret_cast<uint2 *>(base + im.o_att);
    p.hll = reinterpret_cast<uint2 *>(base + im.o_h);
    p.epoch = reinterpret_cast<uint32_t *>(base + im.o_epoch);
    p.lm_part = reinterpret_cast<unsigned long long *>(base + im.o_lm);
    p.lm_cand = reinterpret_cast<unsigned long long *>(base + im.o_cand);
    p.top_k = 0;
    p.top_p = 1.f;
    p.ctr = reinterpret_cast<uint32_t *>(base + im.o_ctr);
    p.exit_ctr = reinterpret_cast<uint32_t *>(base + im.o_exit);
    p.status = reinterpret_cast<int32_t *>(base + im.o_status);
    p.abort_flag = reinterpret_cast<int32_t *>(base + im.o_abort);
    p.rope = reinterpret_cast<const float *>(base + im.o_rope);
    p.instr = reinterpret_cast<const Instr *>(base + im.o_instr);
    p.q_begin = reinterpret_cast<const int32_t *>(base + im.o_qbeg);
    p.n_ranges = im.n_ranges;
    p.ranges = reinterpret_cast<const unsigned long long *>(base + im.o_ranges);
    p.dbg = reinterpret_cast<unsigned long long *>(base + im.o_dbg);
    p.timeout_ns = 2000000000ull;
    p.max_inflight = 3;
    if (const char *env = getenv("MK_MAX_INFLIGHT")) p.max_inflight = atoi(env);
    if (p.max_inflight < 1) p.max_inflight = 1;
    if (p.max_inflight > mk::kPages) p.max_inflight = mk::kPages;
    p.poll_inflight = 2;  // while consumers poll, fewer tiles in flight so their loads do not queue behind tile data
    p.l2_tiles = 0;
    if (const char *env = getenv("MK_L2_TILES")) p.l2_tiles = atoi(env);
    if (p.l2_tiles < 0) p.l2_tiles = 0;
    if (const char *env = getenv("MK_POLL_INFLIGHT")) p.poll_inflight = atoi(env);
    if (p.poll_inflight < 1) p.poll_inflight = 1;
    if (p.poll_inflight > p.max_inflight) p.poll_inflight = p.max_inflight;
}

int upload_image(const Image &im, const mk_config *config, const mk_weights *w,
                 const mk_kv_cache *kv, char *base, cudaStream_t s, const void *lm_w) {
    const mk_config &c = *config;
    const int L = c.n_layers, d = c.d_model, Hq = c.n_heads, Hkv = c.n_kv_heads, hd = c.head_dim,
              F = c.ffn_dim, V = c.vocab;
    // valid byte ranges for the address self-checks of an MK_CHECKED build
    std::vector<unsigned long long> ranges;
    auto add_range = [&](const void *ptr, size_t bytes) {
        ranges.push_back((unsigned long long)(uintptr_t)ptr);
        ranges.push_back((unsigned long long)(uintptr_t)ptr + bytes);
    };
    const size_t kv_bytes = (size_t)L * c.max_batch * Hkv * c.max_seq * hd * 2;
    add_range(base, im.total);
    add_range(kv->k, kv_bytes);
    add_range(kv->v, kv_bytes);
    add_range(w->embed, (size_t)V * d * 2);
    add_range(w->final_norm, (size_t)d * 2);
    add_range(lm_w, lm_w ? (size_t)V * d * 2 : 0);  // (an empty range when absent)
    const int qd = Hq * hd, kvd = Hkv * hd;
    for (int l = 0; l < L; ++l) {
        const mk_layer_weights &lw = w->layers[l];
        add_range(lw.attn_norm, (size_t)d * 2);
        add_range(lw.wq, (size_t)qd * d * 2);
        add_range(lw.wk, (size_t)kvd * d * 2);
        add_range(lw.wv, (size_t)kvd * d * 2);
        add_range(lw.wo, (size_t)d * qd * 2);
        add_range(lw.mlp_norm, (size_t)d * 2);
        add_range(lw.w_gate, (size_t)F * d * 2);
        add_range(lw.w_up, (size_t)F * d * 2);
        add_range(lw.w_down, (size_t)d * F * 2);
    }
    struct Up {
        size_t off;
        const void *src;
        size_t bytes;
    } ups[] = {
        {im.o_ranges, ranges.data(), sizeof(unsigned long long) * ranges.size()},
        {im.o_layers, im.lws.data(), sizeof(mk::LayerW) * im.lws.size()},
        {im.o_rope, im.rope.data(), sizeof(float) * im.rope.size()},
        {im.o_instr, im.flat.data(), sizeof(Instr) * im.flat.size()},
        {im.o_qbeg, im.qbeg.data(), sizeof(int32_t) * im.qbeg.size()},
    };
    cudaError_t e = cudaMemsetAsync(base, 0, im.total, s);
    for (const Up &u : ups)
        if (e == cudaSuccess) e = cudaMemcpyAsync(base + u.off, u.src, u.bytes, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "uploading the plan");
    return MK_OK;
}

int launch_step(const mk::Params &base, int n_sm, int n_stages, int32_t token,
                const int32_t *d_token, int32_t position, float *out_logits, int32_t *out_token,
                cudaStream_t stream, bool unfused, const int32_t *d_pos, int32_t bslot) {
    mk::Params p = base;
    p.token = token;
    p.d_token = d_token;
    p.pos = position;
    p.d_pos = d_pos;
    p.bslot = bslot;
    p.out_logits = out_logits;
    p.out_token = out_token;
    cudaError_t e;
    if (!unfused) {
        p.stage_lo = 0;
        p.stage_hi = n_stages;
        p.reset_at_exit = 1;
        e = mk_kernel_launch(&p, n_sm, 1, stream);
        if (e == cudaErrorCooperativeLaunchTooLarge)
            return fail(MK_ERR_LAUNCH, "persistent grid cannot be co-resident on this device");
        if (e != cudaSuccess) return cuda_fail(e, "megakernel launch");
        return MK_OK;
    }
    for (int s = 0; s < n_stages; ++s) {
        p.stage_lo = s;
        p.stage_hi = s + 1;
        p.reset_at_exit = (s == n_stages - 1);
        e = mk_kernel_launch(&p, n_sm, 0, stream);
        if (e != cudaSuccess) return cuda_fail(e, "stage launch");
    }
    return MK_OK;
}

int set_error(int code, const char *msg) { return fail(code, msg); }

}  // namespace mkint

struct mk_handle {
    mk_config cfg;
    mkint::Image im;
    int device = 0;
    mk::Params base{};     // everything but the per-step fields
    void *dev_mem = nullptr;
    int32_t *d_tok_in = nullptr;   // host path: token staged here
    int32_t *d_tok_out = nullptr;  // host path: greedy token
    float *d_logits = nullptr;     // host path: logits
    size_t zero_bytes = 0;         // counters .. debug record
    unsigned long long timeout_ns = 2000000000ull;
    long long *d_trace = nullptr;
    int trace_cap = 0;
    bool trace_on = false;
    bool trace_batch = false;  // the last traced launch ran the batched image
    float inv_temp = 0.f;      // sampling (mk_set_sampling); 0: greedy
    uint64_t seed = 0;
    int32_t top_k = 0;         // filtered draw (mk_set_sampling_filter); 0: off
    float top_p = 1.f;
    // batched steps of all max_batch sequences in one launch (max_batch > 1 and
    // a model the batched instances support), with their own scratch
    bool has_batch = false;
    mkint::Image bim;
    mk::Params bbase{};
    void *bdev_mem = nullptr;
    void *w16 = nullptr;  // fp16 copies of the GEMV weights (batched steps)
    size_t bzero_bytes = 0;
    // the batched LM head, after the launch on the tensor cores: the bf16
    // embedding's tensor map, the final norm's hi / lo terms [2][max_batch][d],
    // the contraction's wait status, and the logits [max_batch][V] and draw
    // scratch that the step uses when the caller asks for no logits
    CUtensorMap emb_map;
    void *blm_mem = nullptr;
    uint16_t *blm_hi = nullptr, *blm_lo = nullptr;
    int *blm_err = nullptr;
    float *bf_logits = nullptr;
    unsigned long long *bf_lists = nullptr;
    // multi-token prefill (mk_prefill): tensor maps of the weights, made on
    // the first call, and scratch for the largest prompt so far
    bool pf_ready = false;
    mkpf::Model pf_model;
    mkpf::Scratch pf;
    void *pf_mem = nullptr;
    // a sampled draw of the prefill's last position: its logits (when the
    // caller asks for none) and the candidate lists / slice keys
    float *pd_logits = nullptr;
    unsigned long long *pd_lists = nullptr;
};

namespace {

// The last LM-head block gathers and sorts up to n_lm * kMaxTopK candidate
// keys in its page ring, padded to a power of two: at most 16384 (128 KB).
bool filter_in_kernel(const mk_handle *h) { return h->base.n_lm * mk::kMaxTopK <= 16384; }

int launch(mk_handle *h, int32_t token, const int32_t *d_token, int32_t position, float *out_logits,
           int32_t *out_token, cudaStream_t stream, bool unfused, const int32_t *d_pos = nullptr,
           int32_t bslot = 0) {
    if (!h) return fail(MK_ERR_INVALID_ARG, "handle is NULL");
    if (!out_token) return fail(MK_ERR_INVALID_ARG, "out_token is NULL");
    if (!d_pos && (position < 0 || position >= h->cfg.max_seq))
        return fail(MK_ERR_INVALID_ARG, "position outside [0, max_seq)");
    if (!d_token && (token < 0 || token >= h->cfg.vocab))
        return fail(MK_ERR_INVALID_ARG, "token_id outside [0, vocab)");
    cudaError_t e = cudaSetDevice(h->device);
    if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
    mk::Params p = h->base;
    p.timeout_ns = h->timeout_ns;
    p.trace = h->trace_on ? h->d_trace : nullptr;
    p.trace_cap = h->trace_cap;
    p.inv_temp = h->inv_temp;
    p.seed_lo = (uint32_t)(h->seed & 0xFFFFFFFFu);
    p.seed_hi = (uint32_t)(h->seed >> 32);
    // a filter set with only top_p takes the nucleus among the kMaxTopK best
    const bool filtered = h->inv_temp > 0.f && (h->top_k > 0 || h->top_p < 1.f);
    const int K = h->top_k > 0 ? h->top_k : mk::kMaxTopK;
    p.top_k = filtered ? K : 0;
    p.top_p = h->top_p;
    // More LM-head blocks than the last block can sort the candidates of:
    // the launch picks greedily and writes the logits, and the filter
    // kernels of the batched step draw the token after it (same noise:
    // this step's position and slot).
    const bool after = filtered && !filter_in_kernel(h);
    float *logits = out_logits;
    if (after) {
        p.top_k = 0;
        p.inv_temp = 0.f;
        if (!logits) logits = h->d_logits;
    }
    if (h->trace_on) h->trace_batch = false;
    const int rc = mkint::launch_step(p, h->im.n_sm, h->im.n_stages, token, d_token, position, logits, out_token,
                                      stream, unfused, d_pos, bslot);
    if (rc || !after) return rc;
    e = mk_filtered_draw_batch(logits, 1, h->cfg.vocab, K, h->top_p, h->inv_temp, d_pos, d_pos ? 0 : position, bslot,
                               h->seed, h->pd_lists, out_token, stream);
    if (e != cudaSuccess) return cuda_fail(e, "filtered draw");
    return MK_OK;
}

}  // namespace

extern "C" {

const char *mk_last_error(void) { return g_err.c_str(); }

int mk_plan_inspect(const mk_config *config, int32_t n_sm, int32_t *out_instr, int32_t cap,
                    int32_t *out_queue_len, int32_t *out_n_counters) {
    Plan P;
    int rc = MK_ERR_UNSUPPORTED;
    if (config && config->max_batch > 1) rc = build_plan(config, n_sm, P, config->max_batch);
    if (rc) rc = build_plan(config, n_sm, P, 1);
    if (rc) return rc;
    const size_t n = P.n_instr();
    if (out_queue_len)
        for (int s = 0; s < n_sm; ++s) out_queue_len[s] = (int32_t)P.q[s].size();
    if (out_n_counters) *out_n_counters = P.cl.total;
    if (out_instr) {
        if ((size_t)cap < n) return fail(MK_ERR_INVALID_ARG, "cap smaller than the plan");
        size_t k = 0;
        for (int s = 0; s < n_sm; ++s)
            for (const Instr &in : P.q[s]) std::memcpy(out_instr + 16 * (k++), &in, sizeof(Instr));
    }
    return (int)n;
}

int mk_create(const mk_config *config, const mk_weights *w, const mk_kv_cache *kv,
              mk_handle **out) {
    if (!out) return fail(MK_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    int rc = mkint::check_inputs(config, w, kv);
    if (rc) return rc;
    int dev = 0, n_sm = 0;
    rc = mkint::check_device(&dev, &n_sm);
    if (rc) return rc;
    mk_handle *h = new (std::nothrow) mk_handle();
    if (!h) return fail(MK_ERR_NOMEM, "host allocation failed");
    h->cfg = *config;
    h->device = dev;
    rc = mkint::make_image(config, w, n_sm, h->im);
    if (rc) {
        delete h;
        return rc;
    }
    cudaError_t e = cudaMalloc(&h->dev_mem, h->im.total);
    if (e != cudaSuccess) {
        delete h;
        return cuda_fail(e, "cudaMalloc(scratch)");
    }
    char *base = static_cast<char *>(h->dev_mem);
    rc = mkint::upload_image(h->im, config, w, kv, base, nullptr);
    if (rc) {
        cudaFree(h->dev_mem);
        delete h;
        return rc;
    }
    mkint::fill_params(h->im, config, w, kv, base, h->base);
    if (config->max_batch > 1 && config->max_batch <= mk::kMaxBatch &&
        mkint::make_image(config, w, n_sm, h->bim, config->max_batch) == MK_OK) {
        // the batched step runs its GEMVs on fp16 copies of the weights
        const mk_config &c = *config;
        const size_t d = c.d_model, qd = (size_t)c.n_heads * c.head_dim, kvd = (size_t)c.n_kv_heads * c.head_dim,
                     F = c.ffn_dim;
        const size_t per_layer = qd * d + 2 * kvd * d + d * qd + 2 * F * d + d * F;
        const size_t n16 = per_layer * c.n_layers;  // the LM head runs on the bf16 embedding (tensor cores)
        std::vector<mk_layer_weights> lw16(c.n_layers);
        mk_weights w16 = *w;
        // the copy is exact for magnitudes in fp16's normal range; a weight
        // beyond fp16's largest finite value would become an infinity, so
        // such a model keeps sequence-by-sequence batches
        unsigned long long *d_oor = nullptr;
        e = cudaMalloc(&h->w16, n16 * 2 + 256);
        if (e == cudaSuccess) {
            d_oor = reinterpret_cast<unsigned long long *>(static_cast<char *>(h->w16) + ((n16 * 2 + 255) & ~size_t(255)));
            e = cudaMemset(d_oor, 0, sizeof(unsigned long long));
        }
        if (e == cudaSuccess) {
            uint16_t *dst = static_cast<uint16_t *>(h->w16);
            auto copy = [&](const void *src, size_t n) -> const void * {
                uint16_t *at = dst;
                if (e == cudaSuccess) e = mk_convert_bf16_f16(src, at, n, d_oor, nullptr);
                dst += n;
                return at;
            };
            for (int l = 0; l < c.n_layers; ++l) {
                const mk_layer_weights &a = w->layers[l];
                mk_layer_weights &b = lw16[l];
                b = a;
                b.wq = copy(a.wq, qd * d);
                b.wk = copy(a.wk, kvd * d);
                b.wv = copy(a.wv, kvd * d);
                b.wo = copy(a.wo, d * qd);
                b.w_gate = copy(a.w_gate, F * d);
                b.w_up = copy(a.w_up, F * d);
                b.w_down = copy(a.w_down, d * F);
            }
            if (e == cudaSuccess) e = cudaDeviceSynchronize();
            unsigned long long oor = 0;
            if (e == cudaSuccess) e = cudaMemcpy(&oor, d_oor, sizeof oor, cudaMemcpyDeviceToHost);
            if (e == cudaSuccess && oor != 0) e = cudaErrorInvalidValue;  // out of fp16 range: no fused batches
            w16.layers = lw16.data();
            // the image's layer table points at the copies
            for (int l = 0; l < c.n_layers; ++l) {
                const mk_layer_weights &b = lw16[l];
                h->bim.lws[l] = {(const uint16_t *)b.attn_norm, (const uint16_t *)b.wq, (const uint16_t *)b.wk,
                                 (const uint16_t *)b.wv, (const uint16_t *)b.wo, (const uint16_t *)b.mlp_norm,
                                 (const uint16_t *)b.w_gate, (const uint16_t *)b.w_up, (const uint16_t *)b.w_down};
            }
        }
        if (e == cudaSuccess) e = cudaMalloc(&h->bdev_mem, h->bim.total);
        // the LM head's block: hi | lo | logits | draw scratch | status
        const size_t B = c.max_batch, V = c.vocab;
        const size_t o_lo = B * d * 2, o_lg = (2 * B * d * 2 + 255) & ~size_t(255),
                     o_ls = (o_lg + B * V * 4 + 255) & ~size_t(255),
                     o_er = o_ls + sizeof(unsigned long long) * mk_filter_lists_keys((int)B, (int)V);
        if (e == cudaSuccess && (d % 64 || !mkpf::encode_weight_map(&h->emb_map, w->embed, (int)V, (int)d)))
            e = cudaErrorInvalidValue;  // no tensor map of the embedding: no fused batches
        if (e == cudaSuccess) e = cudaMalloc(&h->blm_mem, o_er + sizeof(int));
        if (e == cudaSuccess) {
            char *m = static_cast<char *>(h->blm_mem);
            h->blm_hi = reinterpret_cast<uint16_t *>(m);
            h->blm_lo = reinterpret_cast<uint16_t *>(m + o_lo);
            h->bf_logits = reinterpret_cast<float *>(m + o_lg);
            h->bf_lists = reinterpret_cast<unsigned long long *>(m + o_ls);
            h->blm_err = reinterpret_cast<int *>(m + o_er);
            e = cudaMemset(h->blm_err, 0, sizeof(int));
        }
        if (e != cudaSuccess) {
            // no room for the batched step, or a weight beyond fp16's range:
            // batches run sequence by sequence
            cudaGetLastError();
            if (h->w16) cudaFree(h->w16);
            if (h->bdev_mem) cudaFree(h->bdev_mem);
            if (h->blm_mem) cudaFree(h->blm_mem);
            h->w16 = nullptr;
            h->bdev_mem = nullptr;
            h->blm_mem = nullptr;
            h->blm_hi = h->blm_lo = nullptr;
            h->bf_logits = nullptr;
            h->bf_lists = nullptr;
            h->blm_err = nullptr;
        } else {
            char *bb = static_cast<char *>(h->bdev_mem);
            rc = mkint::upload_image(h->bim, config, &w16, kv, bb, nullptr, nullptr);
            if (rc) {
                cudaFree(h->bdev_mem);
                cudaFree(h->blm_mem);
                cudaFree(h->w16);
                cudaFree(h->dev_mem);
                delete h;
                return rc;
            }
            mkint::fill_params(h->bim, config, &w16, kv, bb, h->bbase);
            h->bbase.lm_w = nullptr;  // no LM-head instructions in the batched plan
            h->bzero_bytes = h->bim.o_zero_end - h->bim.o_ctr;
            h->has_batch = true;
        }
    }
    fail(MK_OK, "");  // a model without batched instances is not an error
    h->d_tok_in = reinterpret_cast<int32_t *>(base + h->im.o_tin);
    h->d_tok_out = reinterpret_cast<int32_t *>(base + h->im.o_tout);
    h->d_logits = reinterpret_cast<float *>(base + h->im.o_logits);
    h->zero_bytes = h->im.o_zero_end - h->im.o_ctr;
    if (getenv("MK_LOG")) {
        size_t mx = 0, mn = (size_t)-1;
        for (int q : h->im.qlen) { mx = std::max(mx, (size_t)q); mn = std::min(mn, (size_t)q); }
        fprintf(stderr, "[mk] plan: %d SMs, %zu instructions (%zu..%zu per SM), %d splits, %zu scratch bytes\n",
                h->im.n_sm, h->im.n_instr, mn, mx, h->base.S, h->im.total);
    }
    *out = h;
    return MK_OK;
}

int mk_decode_step(mk_handle *h, int32_t token_id, int32_t position, float *out_logits,
                   int32_t *out_token, void *stream) {
    return launch(h, token_id, nullptr, position, out_logits, out_token, (cudaStream_t)stream, false);
}

int mk_decode_step_dev(mk_handle *h, const int32_t *d_token_id, int32_t position, float *out_logits,
                       int32_t *out_token, void *stream) {
    if (!d_token_id) return fail(MK_ERR_INVALID_ARG, "d_token_id is NULL");
    return launch(h, 0, d_token_id, position, out_logits, out_token, (cudaStream_t)stream, false);
}

int mk_decode_step_batch(mk_handle *h, const int32_t *d_tokens, const int32_t *d_positions, int32_t batch,
                         float *out_logits, int32_t *out_tokens, void *stream) {
    if (!h) return fail(MK_ERR_INVALID_ARG, "handle is NULL");
    if (!d_tokens || !d_positions || !out_tokens)
        return fail(MK_ERR_INVALID_ARG, "d_tokens, d_positions and out_tokens must not be NULL");
    if (batch < 1 || batch > h->cfg.max_batch) return fail(MK_ERR_INVALID_ARG, "batch outside [1, max_batch]");
    const bool filtered = h->inv_temp > 0.f && (h->top_k > 0 || h->top_p < 1.f);
    if (h->has_batch && batch == h->cfg.max_batch) {
        // All sequences in one launch through the last layer: every weight
        // tile read once for all of them. Then the LM head as one tensor-core
        // contraction over the bf16 embedding (final RMSNorm first, as hi /
        // lo bf16 terms) and every sequence's token drawn from its logits.
        cudaError_t e = cudaSetDevice(h->device);
        if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
        const cudaStream_t s = (cudaStream_t)stream;
        const int V = h->cfg.vocab, d = h->cfg.d_model;
        float *logits = out_logits ? out_logits : h->bf_logits;
        mk::Params p = h->bbase;
        p.timeout_ns = h->timeout_ns;
        p.trace = h->trace_on ? h->d_trace : nullptr;
        p.trace_cap = h->trace_cap;
        if (h->trace_on) h->trace_batch = true;
        const int rc = mkint::launch_step(p, h->bim.n_sm, h->bim.n_stages, 0, d_tokens, 0, nullptr, out_tokens, s,
                                          false, d_positions, 0);
        if (rc) return rc;
        e = mk_batch_final_norm(reinterpret_cast<const float *>(h->bbase.xll), batch, d, h->bbase.final_norm,
                                h->cfg.rms_eps, h->blm_hi, h->blm_lo, s);
        if (e == cudaSuccess)
            e = mkpf::gemm(h->emb_map, h->blm_hi, h->blm_lo, V, batch, d, logits, V, nullptr, nullptr, 0, h->blm_err,
                           h->im.n_sm, s, mkpf::NormOut{});
        if (e != cudaSuccess) return cuda_fail(e, "LM head of the batch");
        // a filter set with only top_p takes the nucleus among the kMaxTopK best
        e = filtered ? mk_filtered_draw_batch(logits, batch, V, h->top_k > 0 ? h->top_k : mk::kMaxTopK, h->top_p,
                                              h->inv_temp, d_positions, 0, 0, h->seed, h->bf_lists, out_tokens, s)
                     : mk_sampled_draw_batch(logits, batch, V, h->inv_temp, d_positions, 0, h->seed, h->bf_lists,
                                             out_tokens, s);
        if (e != cudaSuccess) return cuda_fail(e, "draw of the batch");
        return MK_OK;
    }
    for (int32_t b = 0; b < batch; ++b) {
        const int rc = launch(h, 0, d_tokens + b, 0, out_logits ? out_logits + (size_t)b * h->cfg.vocab : nullptr,
                              out_tokens + b, (cudaStream_t)stream, false, d_positions + b, b);
        if (rc) return rc;
    }
    return MK_OK;
}

int mk_decode_step_unfused(mk_handle *h, int32_t token_id, int32_t position, float *out_logits,
                           int32_t *out_token, void *stream) {
    return launch(h, token_id, nullptr, position, out_logits, out_token, (cudaStream_t)stream, true);
}

int mk_decode_step_host(mk_handle *h, const int32_t *host_token, int32_t position,
                        float *host_logits, int32_t *host_out_token, void *stream) {
    if (!h || !host_token || !host_out_token)
        return fail(MK_ERR_INVALID_ARG, "handle or host token pointer is NULL");
    if (*host_token < 0 || *host_token >= h->cfg.vocab)
        return fail(MK_ERR_INVALID_ARG, "token_id outside [0, vocab)");
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaSetDevice(h->device);
    if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
    // Pinned host buffers that the device can address (cudaHostAlloc'd or
    // registered memory) are used in place: the step reads the token from and
    // writes the next token to host memory over the chip link, with no copy
    // operations on the stream. Other host memory goes through copies.
    const int32_t *tok_in = nullptr;
    int32_t *tok_out = nullptr;
    {
        cudaPointerAttributes ai{}, ao{};
        const cudaError_t qi = cudaPointerGetAttributes(&ai, host_token);
        const cudaError_t qo = qi == cudaSuccess ? cudaPointerGetAttributes(&ao, host_out_token) : cudaSuccess;
        // a failed query only means "not usable in place": clear the error it set
        if (qi != cudaSuccess || qo != cudaSuccess) (void)cudaGetLastError();
        if (qi == cudaSuccess && qo == cudaSuccess && ai.type == cudaMemoryTypeHost && ai.devicePointer &&
            ao.type == cudaMemoryTypeHost && ao.devicePointer) {
            tok_in = static_cast<const int32_t *>(ai.devicePointer);
            tok_out = static_cast<int32_t *>(ao.devicePointer);
        }
    }
    if (!tok_in) {
        e = cudaMemcpyAsync(h->d_tok_in, host_token, sizeof(int32_t), cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, "token upload");
    }
    int rc = launch(h, 0, tok_in ? tok_in : h->d_tok_in, position, host_logits ? h->d_logits : nullptr,
                    tok_out ? tok_out : h->d_tok_out, s, false);
    if (rc) return rc;
    if (!tok_out) {
        e = cudaMemcpyAsync(host_out_token, h->d_tok_out, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) return cuda_fail(e, "token download");
    }
    if (host_logits) {
        e = cudaMemcpyAsync(host_logits, h->d_logits, sizeof(float) * h->cfg.vocab,
                            cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) return cuda_fail(e, "logits download");
    }
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    return MK_OK;
}

int mk_get_status(mk_handle *h) {
    if (!h) return fail(MK_ERR_INVALID_ARG, "handle is NULL");
    cudaError_t e = cudaSetDevice(h->device);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    int32_t st = 0, bst = 0, pst = 0, lst = 0;
    e = cudaMemcpy(&st, h->base.status, sizeof st, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && h->has_batch) e = cudaMemcpy(&bst, h->bbase.status, sizeof bst, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && h->pf.err) e = cudaMemcpy(&pst, h->pf.err, sizeof pst, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && h->blm_err) e = cudaMemcpy(&lst, h->blm_err, sizeof lst, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    if (lst != 0) {
        e = cudaMemset(h->blm_err, 0, sizeof(int));
        if (e != cudaSuccess) return cuda_fail(e, "status reset");
        return fail(MK_ERR_TIMEOUT, "a bounded wait of the batched LM head expired");
    }
    if (pst != 0) {
        e = cudaMemset(h->pf.err, 0, sizeof(int));
        if (e != cudaSuccess) return cuda_fail(e, "status reset");
        if (pst == 2) return fail(MK_ERR_INVALID_ARG, "prompt token outside [0, vocab)");
        return fail(MK_ERR_TIMEOUT, "a bounded wait of the prefill expired");
    }
    if (st == mk::DS_OK && bst == mk::DS_OK) return MK_OK;
    // a failed step leaves counters mid-way: clear them with the status
    e = cudaMemset(h->base.ctr, 0, h->zero_bytes);
    if (e == cudaSuccess && h->has_batch) e = cudaMemset(h->bbase.ctr, 0, h->bzero_bytes);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "status reset");
    if (st == mk::DS_OK) st = bst;
    if (st == mk::DS_BAD_TOKEN) return fail(MK_ERR_INVALID_ARG, "device token outside [0, vocab)");
    if (st == mk::DS_BAD_POS) return fail(MK_ERR_INVALID_ARG, "device position outside [0, max_seq)");
    return fail(MK_ERR_TIMEOUT, "an in-kernel dependency wait timed out");
}

int mk_prefill(mk_handle *h, const int32_t *d_tokens, int32_t n, int32_t start_pos, float *out_logits,
               int32_t *out_token, void *stream) {
    if (!h || !d_tokens || !out_token) return fail(MK_ERR_INVALID_ARG, "handle, d_tokens or out_token is NULL");
    if (n < 1 || start_pos < 0 || (int64_t)start_pos + n > h->cfg.max_seq)
        return fail(MK_ERR_INVALID_ARG, "prompt positions outside [0, max_seq)");
    cudaError_t e = cudaSetDevice(h->device);
    if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
    const mk_config &c = h->cfg;
    const int d = c.d_model, hd = c.head_dim, qd = c.n_heads * hd, kvd = c.n_kv_heads * hd, F = c.ffn_dim;
    if (!h->pf_ready) {
        mkpf::Model &m = h->pf_model;
        m.L = c.n_layers; m.d = d; m.Hq = c.n_heads; m.Hkv = c.n_kv_heads; m.hd = hd; m.F = F; m.V = c.vocab;
        m.max_seq = c.max_seq; m.n_sm = h->im.n_sm; m.eps = c.rms_eps;
        m.embed = h->base.embed;
        m.final_norm = h->base.final_norm;
        m.rope = h->base.rope;
        m.kc = h->base.kc;
        m.vc = h->base.vc;
        m.kv_layer_stride = (size_t)c.max_batch * c.n_kv_heads * c.max_seq * hd;
        m.maps.resize(c.n_layers);
        m.attn_norm.resize(c.n_layers);
        m.mlp_norm.resize(c.n_layers);
        for (int l = 0; l < c.n_layers; ++l) {
            const mk::LayerW &lw = h->im.lws[l];
            mkpf::LayerMaps &lm = m.maps[l];
            m.attn_norm[l] = lw.attn_norm;
            m.mlp_norm[l] = lw.mlp_norm;
            if (!mkpf::encode_weight_map(&lm.wq, lw.wq, qd, d) || !mkpf::encode_weight_map(&lm.wk, lw.wk, kvd, d) ||
                !mkpf::encode_weight_map(&lm.wv, lw.wv, kvd, d) || !mkpf::encode_weight_map(&lm.wo, lw.wo, d, qd) ||
                !mkpf::encode_gated_map(&lm.wg, lw.w_gate, F, d) || !mkpf::encode_gated_map(&lm.wu, lw.w_up, F, d) ||
                !mkpf::encode_weight_map(&lm.wd, lw.w_down, d, F))
                return fail(MK_ERR_UNSUPPORTED, "could not encode the weights' tensor maps");
        }
        h->pf_ready = true;
    }
    if (h->pf.cap < n) {
        // scratch for n tokens: residual and q|k|v (fp32), the hi/lo bf16
        // input of the projections from d or Hq hd columns, and that of the
        // down projection (h = silu(g) * u)
        const size_t kmax = std::max(d, qd), qkv = qd + 2 * kvd;
        // K-split partials: the largest the q/k/v, O and down projections
        // use (gate/up runs in one pass)
        const int nsm = h->im.n_sm;
        const int qkv_rows[3] = {qd, kvd, kvd};
        const size_t work = std::max(std::max(mkpf::gemm_workspace_floats(d, n, qd, nsm, true),
                                              mkpf::gemm_workspace_floats(d, n, F, nsm, true)),
                                     mkpf::gemm_multi_workspace_floats(3, qkv_rows, n, d, nsm));
        // (+ 256 bytes of alignment for each of the 8 pieces)
        const size_t bytes = 4 * (size_t)n * (d + qkv) + 2 * 2 * (size_t)n * (kmax + F) +
                             8 * (size_t)2 * h->im.n_sm + 4 * work + 4 * 512;
        int32_t err_keep = 0;
        if (h->pf.err) cudaMemcpy(&err_keep, h->pf.err, sizeof err_keep, cudaMemcpyDeviceToHost);
        void *mem = nullptr;
        e = cudaMalloc(&mem, bytes);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(prefill scratch)");
        if (h->pf_mem) {
            cudaDeviceSynchronize();
            cudaFree(h->pf_mem);
        }
        h->pf_mem = mem;
        char *b = static_cast<char *>(mem);
        auto take = [&](size_t nbytes) {
            char *at = b;
            b += (nbytes + 255) & ~size_t(255);
            return at;
        };
        mkpf::Scratch &sc = h->pf;
        sc.cap = n;
        sc.X = reinterpret_cast<float *>(take(4 * (size_t)n * d));
        sc.QKV = reinterpret_cast<float *>(take(4 * (size_t)n * qkv));
        sc.Hhi = reinterpret_cast<uint16_t *>(take(2 * (size_t)n * F));
        sc.Hlo = reinterpret_cast<uint16_t *>(take(2 * (size_t)n * F));
        sc.Ahi = reinterpret_cast<uint16_t *>(take(2 * (size_t)n * kmax));
        sc.Alo = reinterpret_cast<uint16_t *>(take(2 * (size_t)n * kmax));
        sc.keys = reinterpret_cast<unsigned long long *>(take(8 * (size_t)2 * h->im.n_sm));
        sc.work = reinterpret_cast<float *>(take(4 * work));
        sc.work_floats = work;
        sc.err = reinterpret_cast<int *>(take(4));
        e = cudaMemcpy(sc.err, &err_keep, sizeof err_keep, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "prefill status");
    }
    // with sampling on, the token of the last position is drawn as the decode
    // step at that position would draw it (same noise, same filter)
    const bool sampled = h->inv_temp > 0.f;
    float *logits = out_logits;
    if (sampled) {
        if (!h->pd_lists) {
            e = cudaMalloc(&h->pd_lists, sizeof(unsigned long long) * mk_filter_lists_keys(1, h->cfg.vocab));
            if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(prefill draw lists)");
        }
        if (!logits && !h->pd_logits) {
            e = cudaMalloc(&h->pd_logits, sizeof(float) * (size_t)h->cfg.vocab);
            if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(prefill logits)");
        }
        if (!logits) logits = h->pd_logits;
    }
    e = mkpf::run(h->pf_model, h->pf, d_tokens, n, start_pos, logits, out_token, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    if (sampled) {
        const int pos = start_pos + n - 1;
        if (h->top_k > 0 || h->top_p < 1.f)
            e = mk_filtered_draw_batch(logits, 1, h->cfg.vocab, h->top_k > 0 ? h->top_k : mk::kMaxTopK, h->top_p,
                                       h->inv_temp, nullptr, pos, 0, h->seed, h->pd_lists, out_token,
                                       (cudaStream_t)stream);
        else
            e = mk_sampled_draw_batch(logits, 1, h->cfg.vocab, h->inv_temp, nullptr, pos, h->seed, h->pd_lists,
                                      out_token, (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, "prefill draw");
    }
    return MK_OK;
}

int mk_set_wait_timeout(mk_handle *h, uint64_t timeout_ns) {
    if (!h || timeout_ns == 0) return fail(MK_ERR_INVALID_ARG, "bad handle or zero timeout");
    h->timeout_ns = timeout_ns;
    return MK_OK;
}

int mk_set_sampling(mk_handle *h, float temperature, uint64_t seed) {
    if (!h) return fail(MK_ERR_INVALID_ARG, "handle is NULL");
    if (!(temperature == temperature) || temperature > 1e30f || temperature < -1e30f)
        return fail(MK_ERR_INVALID_ARG, "temperature is not finite");
    if (temperature > 0.f && 1.0f / temperature > 1e30f) return fail(MK_ERR_INVALID_ARG, "temperature too small");
    h->inv_temp = temperature > 0.f ? 1.0f / temperature : 0.f;
    h->seed = seed;
    return MK_OK;
}

int mk_set_sampling_filter(mk_handle *h, int32_t top_k, float top_p) {
    if (!h) return fail(MK_ERR_INVALID_ARG, "handle is NULL");
    if (top_k < 0 || top_k > mk::kMaxTopK) return fail(MK_ERR_INVALID_ARG, "top_k outside [0, 64]");
    if (!(top_p > 0.f && top_p <= 1.f)) return fail(MK_ERR_INVALID_ARG, "top_p outside (0, 1]");
    // a model whose candidates do not fit the in-kernel sort draws with the
    // filter kernels after the launch: their candidate lists are made here
    if ((top_k > 0 || top_p < 1.f) && !filter_in_kernel(h) && !h->pd_lists) {
        const cudaError_t e = cudaMalloc(&h->pd_lists, sizeof(unsigned long long) * mk_filter_lists_keys(1, h->cfg.vocab));
        if (e != cudaSuccess) {
            h->pd_lists = nullptr;
            return cuda_fail(e, "cudaMalloc(filter lists)");
        }
    }
    h->top_k = top_k;
    h->top_p = top_p;
    return MK_OK;
}

int mk_sampling_noise(int32_t n, int32_t position, int32_t slot, uint64_t seed, const uint32_t *d_words,
                      uint32_t *d_out_words, float *d_out_noise, void *stream) {
    if (n < 0) return fail(MK_ERR_INVALID_ARG, "n must be >= 0");
    if (!d_out_words && !d_out_noise) return fail(MK_ERR_INVALID_ARG, "no output buffer");
    const cudaError_t e = mk_noise_launch(n, position, slot, seed, d_words, d_out_words, d_out_noise,
                                          (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "noise kernel launch");
    return MK_OK;
}

int mk_draw_from_logits(const float *d_logits, int32_t batch, int32_t vocab, float temperature, int32_t top_k,
                        float top_p, const int32_t *d_positions, uint64_t seed, int32_t *d_out_tokens, void *stream) {
    if (!d_logits || !d_positions || !d_out_tokens) return fail(MK_ERR_INVALID_ARG, "NULL pointer");
    if (batch < 1 || vocab < 1) return fail(MK_ERR_INVALID_ARG, "batch and vocab must be >= 1");
    if (!(temperature > 0.f) || !std::isfinite(temperature))
        return fail(MK_ERR_INVALID_ARG, "temperature must be finite and > 0");
    if (top_k < 0 || top_k > mk::kMaxTopK) return fail(MK_ERR_INVALID_ARG, "top_k outside [0, MK_MAX_TOP_K]");
    if (!(top_p > 0.f && top_p <= 1.f)) return fail(MK_ERR_INVALID_ARG, "top_p outside (0, 1]");
    // the kernels' scratch: candidate lists (or slice keys), grown as needed
    static unsigned long long *work = nullptr;
    static size_t have = 0;
    const size_t need = mk_filter_lists_keys(batch, vocab);
    if (need > have) {
        if (work) {
            cudaDeviceSynchronize();
            cudaFree(work);
        }
        work = nullptr;
        have = 0;
        const cudaError_t e = cudaMalloc(&work, need * sizeof(unsigned long long));
        if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(draw scratch)");
        have = need;
    }
    const float inv_temp = 1.0f / temperature;
    const cudaError_t e =
        top_k > 0 || top_p < 1.f
            ? mk_filtered_draw_batch(d_logits, batch, vocab, top_k > 0 ? top_k : mk::kMaxTopK, top_p, inv_temp,
                                     d_positions, 0, 0, seed, work, d_out_tokens, (cudaStream_t)stream)
            : mk_sampled_draw_batch(d_logits, batch, vocab, inv_temp, d_positions, 0, seed, work, d_out_tokens,
                                    (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "draw kernels");
    return MK_OK;
}

int mk_set_trace(mk_handle *h, int32_t enable) {
    if (!h) return fail(MK_ERR_INVALID_ARG, "handle is NULL");
    if (enable && !h->d_trace) {
        int cap = 0;
        for (int q : h->im.qlen) cap = std::max(cap, q);
        if (h->has_batch)
            for (int q : h->bim.qlen) cap = std::max(cap, q);
        cap = std::max(cap, 1);
        cudaError_t e = cudaSetDevice(h->device);
        if (e == cudaSuccess)
            e = cudaMalloc(&h->d_trace, sizeof(long long) * mk::kTraceWords * (size_t)cap * h->im.n_sm);
        if (e == cudaSuccess)
            e = cudaMemset(h->d_trace, 0, sizeof(long long) * mk::kTraceWords * (size_t)cap * h->im.n_sm);
        if (e != cudaSuccess) {
            h->d_trace = nullptr;
            return cuda_fail(e, "trace buffer");
        }
        h->trace_cap = cap;
    }
    h->trace_on = enable != 0;
    return MK_OK;
}

int mk_read_trace(mk_handle *h, int64_t *host_out, int32_t cap) {
    if (!h || cap < 0) return fail(MK_ERR_INVALID_ARG, "bad arguments");
    if (!h->d_trace) return 0;
    const mkint::Image &im = h->trace_batch ? h->bim : h->im;
    if (!host_out) {
        int n = 0;
        for (int s = 0; s < im.n_sm; ++s) n += std::min(im.qlen[s], h->trace_cap);
        return n;
    }
    std::vector<long long> buf(mk::kTraceWords * (size_t)h->trace_cap * im.n_sm);
    cudaError_t e = cudaSetDevice(h->device);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess)
        e = cudaMemcpy(buf.data(), h->d_trace, sizeof(long long) * buf.size(), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "trace read");
    int n = 0;
    for (int s = 0; s < im.n_sm; ++s)
        for (int i = 0; i < im.qlen[s] && i < h->trace_cap; ++i) {
            if (n >= cap) return n;
            std::memcpy(host_out + mk::kTraceWords * (size_t)n,
                        &buf[mk::kTraceWords * ((size_t)s * h->trace_cap + i)],
                        mk::kTraceWords * sizeof(long long));
            ++n;
        }
    return n;
}

int mk_debug_read(mk_handle *h, uint64_t *host_out4) {
    if (!h || !host_out4) return fail(MK_ERR_INVALID_ARG, "bad arguments");
    cudaError_t e = cudaSetDevice(h->device);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess)
        e = cudaMemcpy(host_out4, h->base.dbg, 4 * sizeof(uint64_t), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "debug read");
#ifdef MK_CHECKED
    return 1;
#else
    return 0;
#endif
}

int mk_plan_size(const mk_handle *h, int32_t *n_sm, int32_t *n_instr) {
    if (!h) return fail(MK_ERR_INVALID_ARG, "handle is NULL");
    if (n_sm) *n_sm = h->im.n_sm;
    if (n_instr) *n_instr = (int32_t)h->im.n_instr;
    return MK_OK;
}

void mk_destroy(mk_handle *h) {
    if (!h) return;
    cudaSetDevice(h->device);
    cudaDeviceSynchronize();
    if (h->d_trace) cudaFree(h->d_trace);
    if (h->dev_mem) cudaFree(h->dev_mem);
    if (h->bdev_mem) cudaFree(h->bdev_mem);
    if (h->w16) cudaFree(h->w16);
    if (h->pf_mem) cudaFree(h->pf_mem);
    if (h->blm_mem) cudaFree(h->blm_mem);  // holds bf_logits and bf_lists
    if (h->pd_logits) cudaFree(h->pd_logits);
    if (h->pd_lists) cudaFree(h->pd_lists);
    delete h;
}

}  // extern "C"
