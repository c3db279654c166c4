// mk_prefill.h — host-side interface of the prefill kernels (mk_prefill.cu)
// for the C ABI in mk_host.cpp. Not part of the C ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

namespace mkpf {

// Tensor maps of one layer's projection weights (bf16 [out][in], boxes of
// 64 x 128, 128-byte swizzle; wg and wu boxes of 64 x 64, as the gated
// launch takes 64 rows of each).
struct LayerMaps {
    CUtensorMap wq, wk, wv, wo, wg, wu, wd;
};

// The model as the prefill reads it (device pointers; borrowed).
struct Model {
    int L = 0, d = 0, Hq = 0, Hkv = 0, hd = 0, F = 0, V = 0, max_seq = 0, n_sm = 0;
    float eps = 0.f;
    const uint16_t *embed = nullptr, *final_norm = nullptr;
    std::vector<const uint16_t *> attn_norm, mlp_norm;
    std::vector<LayerMaps> maps;
    const float *rope = nullptr;  // [max_seq][hd/2][2] cos, sin
    uint16_t *kc = nullptr, *vc = nullptr;  // KV cache of batch slot 0 of layer 0
    size_t kv_layer_stride = 0;             // elements from one layer's slot-0 cache to the next
};

// Device scratch for up to `cap` prompt tokens.
struct Scratch {
    int cap = 0;
    float *X = nullptr, *QKV = nullptr;
    uint16_t *Ahi = nullptr, *Alo = nullptr;  // hi / lo terms of a contraction's input [n][<= max(d, Hq hd)]
    uint16_t *Hhi = nullptr, *Hlo = nullptr;  // hi / lo terms of h = silu(g) * u [n][F]
    unsigned long long *keys = nullptr;
    float *work = nullptr;   // K-split partial sums of the contractions
    size_t work_floats = 0;
    int *err = nullptr;  // 0 ok, 1 a bounded wait expired, 2 a token outside [0, vocab)
};

bool encode_weight_map(CUtensorMap *map, const void *w, int rows, int K);
bool encode_gated_map(CUtensorMap *map, const void *w, int rows, int K);  // W_gate / W_up, for gemm_gated

// An RMSNorm formed from a contraction's output rows: hi / lo bf16 terms
// [n][M] of RMSNorm(Y[n]) with gains g (g NULL: none).
struct NormOut {
    const uint16_t *g = nullptr;
    float eps = 0.f;
    uint16_t *hi = nullptr, *lo = nullptr;
};

// Y[n][m] (+)= W[m][.] . (Bhi[n][.] + Blo[n][.]) on the tensor cores, then
// the norm nm of Y's rows (ldy == M); work (work_floats floats) holds K-split
// partial sums (one pass if too small).
cudaError_t gemm(const CUtensorMap &wmap, const void *bhi, const void *blo, int M, int N, int K, float *Y, int ldy,
                 const float *R, float *work, size_t work_floats, int *err, int n_sm, cudaStream_t s,
                 const NormOut &nm);

// hi / lo bf16 terms of h[n][f] = silu(g) * u, g and u the rows f of W_gate
// and W_up (maps from encode_gated_map) times Bhi[n][.] + Blo[n][.]; one
// pass, no K split.
cudaError_t gemm_gated(const CUtensorMap &wg, const CUtensorMap &wu, int F, const void *bhi, const void *blo, int N,
                       int K, uint16_t *hhi, uint16_t *hlo, int *err, int n_sm, cudaStream_t s);

// Floats of K-split workspace gemm() uses for this shape, with or without a
// norm of its output (0: none).
size_t gemm_workspace_floats(int M, int N, int K, int n_sm, bool norm);

// Floats of K-split partials the prefill's q/k/v launch (nseg matrices of M[i]
// rows) leaves for its RoPE pass (0: none).
size_t gemm_multi_workspace_floats(int nseg, const int *M, int N, int K, int n_sm);

// The prompt d_tokens[0 .. n) at positions pos0 .. pos0+n-1 through every
// layer: K/V rows of every position into the cache, logits of the last
// position into out_logits (nullable) and its greedy token into out_token.
cudaError_t run(const Model &m, const Scratch &sc, const int32_t *d_tokens, int n, int pos0, float *out_logits,
                int32_t *out_token, cudaStream_t s);

}  // namespace mkpf
