// mk_plan.h — instruction format, tile geometry and kernel parameters shared
// by the host scheduler (mk_host.cpp) and the persistent interpreter kernel
// (mk_kernel.cu).
//
// The design follows the megakernel article ("Revolution der
// KI-Beschleunigung: Wie ein Low-Latency Megakernel den Llama-1B Turbo
// zündet", dasgeld.co): the host plans one instruction sequence per SM once
// (internal-infrastructure paragraph), the kernel interprets it, and every
// instruction waits for exactly the data it consumes through flags kept in
// global memory (synchronisation paragraph). Here the flag travels inside
// each activation word: an element is stored as {float value, 32-bit tag}
// in one 8-byte write, the tag naming the decode step and the version of the
// tensor, and a consumer polls the words it needs until all carry the tag it
// expects. The plan's per-instruction dependency counts (wait_ctr /
// wait_target) describe the same edges for the host-side validator.
#pragma once
#include <stdint.h>

namespace mk {

// ---- fixed kernel geometry ------------------------------------------------
constexpr int kConsumerWarps = 8;                    // compute warps per CTA
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;      // + one producer (TMA) warp
constexpr int kPageBytes = 32768;                    // one shared-memory page
constexpr int kPages = 6;                            // pages in the ring
constexpr int kRedCap = 2048;                        // floats of per-row partials
constexpr int kBatchAcc = 8192;                      // floats of the batched GEMV's accumulators (xbuf + red)
constexpr int kXbufFloats = 6144;                    // staged input (4096 fp32 + 4096 bf16 gains) / attention scratch
constexpr int kMaxStaged = 4096;                     // max normed input length staged with its gains
constexpr int kMaxStagedLong = 8192;                 // max un-normed input length (down projection)
constexpr int kResidFloats = 256;                    // residual rows of one O-proj / down instruction
constexpr int kDredFloats = 256;                     // per-row partials of one down instruction
constexpr int kMaxBatch = 8;                         // sequences of one batched step
constexpr int kMaxG = 8;                             // max query heads per kv head (1,2,3,4,6,8)
constexpr int kTraceWords = 8;                       // int64 per trace record
constexpr int kMinSplitTiles = 4;                    // an attention split gets >= 4 KV tiles
constexpr int kMergeBatch = 1;                       // splits read together by the merge
constexpr int kMaxTopK = 64;                         // candidates kept per LM-head block (top-k / top-p)

constexpr int kSmemPages = 0;
constexpr int kSmemXbuf = kSmemPages + kPages * kPageBytes;
// The partials buffer `red` is the top 8 KB of the 32 KB staging area: ops
// that stage at most kXbufFloats floats use both; the down projection stages
// up to 8192 floats over both and keeps its partials in `dred`.
constexpr int kSmemRed = kSmemXbuf + kXbufFloats * 4;
constexpr int kSmemResid = kSmemXbuf + kMaxStagedLong * 4;
constexpr int kSmemDred = kSmemResid + kResidFloats * 4;
constexpr int kSmemBars = kSmemDred + kDredFloats * 4;
constexpr int kSmemMisc = kSmemBars + 2 * kPages * 8;
constexpr int kSmemParams = kSmemMisc + 256;      // shared copy of the launch parameters
constexpr int kParamsSlot = 640;
constexpr int kSmemBytes = kSmemParams + kParamsSlot;
static_assert(kSmemXbuf + kBatchAcc * 4 <= kSmemResid, "batched accumulators overlap the residual rows");
static_assert(kSmemBytes <= 232448, "shared memory of one CTA exceeds 227 KB");
static_assert(16384 * 8 <= kPages * kPageBytes, "the filtered draw sorts up to 16384 keys in the page ring");

// ---- opcodes ------------------------------------------------------------
enum Op : int32_t {
    OP_QKV = 1,     // rows of Wq|Wk|Wv on RMSNorm(x): writes raw q,k,v
    OP_ATTN = 2,    // one KV split of one kv head: RoPE, KV append, partial softmax, LSE merge
    OP_OPROJ = 3,   // rows of Wo on the attention output, + residual
    OP_GATEUP = 4,  // rows of Wg and Wu on RMSNorm(x), silu(g)*u
    OP_DOWN = 5,    // rows of Wd on h, + residual
    OP_LMHEAD = 6,  // rows of the tied embedding on RMSNorm(x), logits + block argmax
};
constexpr int kStagesPerLayer = 5;

// One instruction = 16 int32 (64 bytes).
struct alignas(16) Instr {
    int32_t op, layer;
    int32_t a0, a1;         // GEMV: first row, row count.  ATTN: kv head, split
    int32_t mat;            // QKV: 0 q, 1 k, 2 v
    int32_t wait_ctr;       // counter to wait on (-1: none)
    int32_t wait_target;    // ... until it reaches this value
    int32_t sig_ctr, sig_n; // counters [sig_ctr, sig_ctr+sig_n) to bump by 1 when done
    int32_t stage;          // topological stage (QKV(l)=5l ... LMHEAD=5L)
    int32_t slot;           // LMHEAD: argmax partial slot.  ATTN: part of the kv head's query heads
    int32_t bytes_lo, bytes_hi;  // weight bytes streamed (host bookkeeping)
    int32_t pad[3];
};
static_assert(sizeof(Instr) == 64, "Instr must be 64 bytes");

// Tile geometry of one GEMV operand shape (input length K).
// A warp owns rows of a tile (row group rg) and a K-slice (ks):
//   sw = K-slices per row, rw = 8/sw row groups, m rows per warp per tile,
//   rt = rw*m rows per tile, nx = floats of the input each lane keeps.
// Batched steps: tiles hold rt rows x a K-chunk of pad (<= 1024) columns,
// each warp a 128-wide slice of the chunk (kslice) and m = 16 rows; the
// chunks of one row are separate tiles.
struct Geo {
    int32_t K, sw, rw, m, rt, nx, kslice, pad;
};

struct LayerW {
    const uint16_t *attn_norm, *wq, *wk, *wv, *wo, *mlp_norm, *w_gate, *w_up, *w_down;
};

// Counter index layout (all uint32 in one device array).
struct CtrLayout {
    int32_t qkv_grp;   // + l*Hkv + h : QKV instructions of group h done
    int32_t merge;     // + l*Hkv + h : attention splits arrived
    int32_t attn_done; // + l        : kv heads merged
    int32_t oproj_done, gateup_done, down_done;  // + l
    int32_t lm_arrive; // LM-head instructions arrived
    int32_t total;
};

struct Params {
    // shape
    int32_t L, d, Hq, Hkv, hd, F, V, max_seq, max_batch, S, G, ppt;
    int32_t attn_heads;     // query heads of one attention instruction (G, or G/2 when a kv head's
                            // query heads are split over two instructions)
    float eps;
    int32_t n_lm, n_stages;
    Geo geo_qkv, geo_o, geo_gu, geo_down, geo_lm;
    CtrLayout cl;
    // weights (borrowed)
    const uint16_t *embed, *final_norm;
    const uint16_t *lm_w;  // LM-head weight rows: the tied embedding (batched steps: its fp16 copy)
    const LayerW *layers;   // device array [L]
    uint16_t *kc, *vc;      // KV caches
    // scratch (library-owned); activations are tagged words {value, tag}
    uint2 *xll;             // [d] residual stream (versions 2l+1 after O-proj l, 2l+2 after down l)
    uint2 *qkvll;           // [L][(Hq+2Hkv)*hd] raw projections
    uint2 *partll;          // [L][Hq][S][hd+2] split partials (o, m, l)
    uint2 *attll;           // [L][Hq*hd] attention output
    uint2 *hll;             // [L][F] silu(g)*u
    uint32_t *epoch;        // decode-step counter (tags carry it); advanced by the last CTA
    unsigned long long *lm_part;  // [n_lm] packed (value, ~index)
    uint32_t *ctr;          // dependency counters
    uint32_t *exit_ctr;     // CTAs done with the step
    int32_t *status;        // 0 ok, else error code (sticky until read)
    int32_t *abort_flag;
    const float *rope;      // [max_seq][hd/2][2] cos, sin
    const Instr *instr;     // flat queues
    const int32_t *q_begin; // [n_sm][n_stages+1] first instruction index with stage >= s
    // this launch
    int32_t stage_lo, stage_hi, reset_at_exit;
    int32_t token;
    const int32_t *d_token; // if non-null, overrides token
    int32_t pos;
    const int32_t *d_pos;   // if non-null, overrides pos (read once at the start of the step)
    int32_t bslot;          // batch slot of the KV cache this step reads and appends to
    // batched step (nb > 1): d_token and d_pos hold nb entries; sequence b
    // uses KV slot b and the b-th row of every activation buffer
    int32_t nb;
    int32_t posb[kMaxBatch];
    float *out_logits;      // nullable
    int32_t *out_token;
    // sampling (inv_temp > 0): the token is argmax_i(logit_i * inv_temp + g_i)
    // with Gumbel noise g_i from Philox4x32-10 keyed by the seed; 0: greedy
    float inv_temp;
    uint32_t seed_lo, seed_hi;
    // top-k / top-p filtering of the draw (inv_temp > 0 and top_k > 0): the
    // top_k best logits, then the shortest prefix of them whose softmax mass
    // reaches top_p; lm_cand holds each LM-head block's kMaxTopK best keys
    int32_t top_k;
    float top_p;
    unsigned long long *lm_cand;  // [n_lm][kMaxTopK]
    unsigned long long timeout_ns;
    long long *trace;       // nullable: [n_sm][trace_cap][kTraceWords]
    int32_t trace_cap;
    int32_t max_inflight;             // tiles per SM whose copies may be outstanding at once
    int32_t poll_inflight;            // ... while the consumers poll for an instruction's input
    int32_t l2_tiles;                 // tiles beyond the smem ring the producer may pull into L2 while it waits
    // address self-checks (only read by a build with MK_CHECKED defined)
    int32_t n_ranges;
    const unsigned long long *ranges;  // [n_ranges][2] valid [begin, end) byte ranges
    unsigned long long *dbg;           // first violation: site, address, bytes, block/thread
};
static_assert(sizeof(Params) <= kParamsSlot, "Params must fit its shared-memory slot");

// Device status codes written to *status.
enum DevStatus : int32_t { DS_OK = 0, DS_TIMEOUT = 1, DS_BAD_TOKEN = 2, DS_BAD_POS = 3 };

}  // namespace mk
