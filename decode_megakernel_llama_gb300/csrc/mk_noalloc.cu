// mk_noalloc.cu — the decode step for callers that cannot allocate device
// memory.
//
// Some callers cannot call cudaMalloc: code that runs under a memory budget
// enforced by a host framework with its own pool, plugins that may only use
// the buffers they are handed, or code paths where an allocation would
// synchronise the device at a bad time. mk_decode_step_noalloc serves them:
// it runs the same persistent megakernel as mk_decode_step, but keeps the
// kernel's scratch (instruction queues, dependency counters, activations,
// attention partials, RoPE table) in one file-scope device array instead of
// memory from cudaMalloc. The caller still passes the weights, the KV cache
// and the output buffers.
//
// The array is kNoAllocScratchBytes (16 MiB) and exists on every GPU that
// loads this library, from load until process exit.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "mk_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

// Host code must not use this name as an address: it is the host-side
// shadow of the symbol. The device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct DeviceSlot {
    bool ready = false;
    char *base = nullptr;             // device address of g_noalloc_scratch on this device
    std::vector<unsigned char> key;   // the inputs the resident plan was built for
    mkint::Image im;
    mk::Params params{};
};

std::mutex g_mu;
DeviceSlot g_slots[kMaxDevices];

template <class T>
void put(std::vector<unsigned char> &k, const T &v) {
    const unsigned char *b = reinterpret_cast<const unsigned char *>(&v);
    k.insert(k.end(), b, b + sizeof(T));
}

void make_key(const mk_config *c, const mk_weights *w, const mk_kv_cache *kv, int n_sm,
              std::vector<unsigned char> &k) {
    k.clear();
    put(k, *c);
    put(k, n_sm);
    put(k, w->embed);
    put(k, w->final_norm);
    for (int l = 0; l < c->n_layers; ++l) put(k, w->layers[l]);
    put(k, kv->k);
    put(k, kv->v);
}

}  // namespace

extern "C" int mk_decode_step_noalloc(const mk_config *config, const mk_weights *weights,
                                      const mk_kv_cache *kv, int32_t token_id, int32_t position,
                                      float *out_logits, int32_t *out_token, void *stream) {
    int rc = mkint::check_inputs(config, weights, kv);
    if (rc) return rc;
    if (!out_token) return mkint::set_error(MK_ERR_INVALID_ARG, "out_token is NULL");
    if (position < 0 || position >= config->max_seq)
        return mkint::set_error(MK_ERR_INVALID_ARG, "position outside [0, max_seq)");
    if (token_id < 0 || token_id >= config->vocab)
        return mkint::set_error(MK_ERR_INVALID_ARG, "token_id outside [0, vocab)");
    int dev = 0, n_sm = 0;
    rc = mkint::check_device(&dev, &n_sm);
    if (rc) return rc;
    if (dev < 0 || dev >= kMaxDevices)
        return mkint::set_error(MK_ERR_UNSUPPORTED, "device ordinal above 63");
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    std::lock_guard<std::mutex> lock(g_mu);
    DeviceSlot &sl = g_slots[dev];
    if (!sl.ready) {
        // once per device, with that device current
        void *ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || !ptr)
            return mkint::set_error(MK_ERR_CUDA, (std::string("cudaGetSymbolAddress: ") +
                                                  cudaGetErrorString(e)).c_str());
        sl.base = static_cast<char *>(ptr);
        sl.ready = true;
    }
    std::vector<unsigned char> key;
    make_key(config, weights, kv, n_sm, key);
    if (key != sl.key) {
        mkint::Image im;
        rc = mkint::make_image(config, weights, n_sm, im);
        if (rc) return rc;
        if (im.total > kNoAllocScratchBytes)
            return mkint::set_error(
                MK_ERR_INVALID_ARG,
                ("this model needs " + std::to_string(im.total) + " bytes of scratch; the static "
                 "array holds " + std::to_string(kNoAllocScratchBytes) + " (use mk_create)").c_str());
        sl.key.clear();  // a failed upload leaves no valid resident plan
        rc = mkint::upload_image(im, config, weights, kv, sl.base, s);
        if (rc) return rc;
        mkint::fill_params(im, config, weights, kv, sl.base, sl.params);
        sl.im = std::move(im);
        sl.key = std::move(key);
    }
    // Counters, status and abort flag must start at zero; a previous call may
    // have left them mid-way if it hit its wait limit.
    cudaError_t e = cudaMemsetAsync(sl.base + sl.im.o_ctr, 0, sl.im.o_zero_end - sl.im.o_ctr, s);
    if (e != cudaSuccess)
        return mkint::set_error(MK_ERR_CUDA, (std::string("cudaMemsetAsync: ") +
                                              cudaGetErrorString(e)).c_str());
    return mkint::launch_step(sl.params, sl.im.n_sm, sl.im.n_stages, token_id, nullptr, position,
                              out_logits, out_token, s, false);
}
