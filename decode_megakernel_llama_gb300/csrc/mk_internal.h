// mk_internal.h — host-side pieces shared by the handle-based entry points
// (mk_host.cpp) and the allocation-free entry point (mk_noalloc.cu): the
// device image of a plan (layout of one scratch region plus the host arrays
// uploaded into it) and the launch of one step. Not part of the C ABI.
#pragma once
#include <cuda_runtime.h>

#include <memory>
#include <vector>

#include "../../include/mk.h"
#include "mk_plan.h"

namespace mkint {

struct ImageImpl;

struct Image {
    std::shared_ptr<ImageImpl> impl;  // the plan
    int n_sm = 0, n_stages = 0, n_ranges = 0;
    size_t n_instr = 0, total = 0;
    // byte offsets into the scratch region; [o_ctr, o_zero_end) starts at zero
    size_t o_ctr = 0, o_exit = 0, o_status = 0, o_abort = 0, o_dbg = 0, o_zero_end = 0;
    size_t o_epoch = 0, o_layers = 0, o_x = 0, o_qkv = 0, o_part = 0, o_att = 0, o_h = 0, o_lm = 0;
    size_t o_cand = 0, o_tin = 0, o_tout = 0, o_logits = 0, o_rope = 0, o_instr = 0, o_qbeg = 0, o_ranges = 0;
    std::vector<mk::Instr> flat;
    std::vector<int32_t> qbeg;
    std::vector<float> rope;
    std::vector<mk::LayerW> lws;
    std::vector<int> qlen;
};

int check_inputs(const mk_config *config, const mk_weights *w, const mk_kv_cache *kv);
int check_device(int *dev, int *n_sm);
int make_image(const mk_config *config, const mk_weights *w, int n_sm, Image &im, int nb = 1);
// lm_w: a separate copy of the LM-head weights to register for the
// address self-checks (batched steps), or NULL
int upload_image(const Image &im, const mk_config *config, const mk_weights *w,
                 const mk_kv_cache *kv, char *base, cudaStream_t s, const void *lm_w = nullptr);
void fill_params(const Image &im, const mk_config *config, const mk_weights *w,
                 const mk_kv_cache *kv, char *base, mk::Params &p);
int launch_step(const mk::Params &base, int n_sm, int n_stages, int32_t token,
                const int32_t *d_token, int32_t position, float *out_logits, int32_t *out_token,
                cudaStream_t stream, bool unfused, const int32_t *d_pos = nullptr, int32_t bslot = 0);
int set_error(int code, const char *msg);

}  // namespace mkint
