"""Thin ctypes binding of libmk.so (include/mk.h): argument marshalling only.

Every step of the decode path runs in the library's CUDA kernels; this module
only turns torch tensors into device pointers and sizes. If the library is
missing it raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libmk.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "mk.h")

MK_OK = 0
MK_ERR_INVALID_ARG = -1
MK_ERR_CUDA = -2
MK_ERR_LAUNCH = -3
MK_ERR_UNSUPPORTED = -4
MK_ERR_TIMEOUT = -5
MK_ERR_NOMEM = -6
MK_INSTR_WORDS = 16


class MKError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"mk error {code}: {msg}")
        self.code = code


class mk_config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("d_model", ctypes.c_int32),
                ("n_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("ffn_dim", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("max_seq", ctypes.c_int32),
                ("max_batch", ctypes.c_int32), ("attn_splits", ctypes.c_int32),
                ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float)]


class mk_layer_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm",
                                               "w_gate", "w_up", "w_down")]


class mk_weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
                ("layers", ctypes.POINTER(mk_layer_weights))]


class mk_kv_cache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p)]


_lib = None
_VP = ctypes.c_void_p
_I32 = ctypes.c_int32
_PI32 = ctypes.POINTER(ctypes.c_int32)


def load(path: str | None = None):
    """Loads libmk.so (built by decode_megakernel_llama_gb300.build). The
    environment variable MK_LIB selects another build of the same library
    (e.g. the address-checked one)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or os.environ.get("MK_LIB") or LIB_PATH
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: run decode_megakernel_llama_gb300.build.build() "
                          "(there is no fallback implementation)")
    L = ctypes.CDLL(path)
    L.mk_last_error.restype = ctypes.c_char_p
    L.mk_create.argtypes = [ctypes.POINTER(mk_config), ctypes.POINTER(mk_weights),
                            ctypes.POINTER(mk_kv_cache), ctypes.POINTER(_VP)]
    L.mk_decode_step.argtypes = [_VP, _I32, _I32, _VP, _VP, _VP]
    L.mk_decode_step_dev.argtypes = [_VP, _VP, _I32, _VP, _VP, _VP]
    L.mk_decode_step_host.argtypes = [_VP, _PI32, _I32, _VP, _PI32, _VP]
    L.mk_decode_step_unfused.argtypes = [_VP, _I32, _I32, _VP, _VP, _VP]
    L.mk_decode_step_batch.argtypes = [_VP, _VP, _VP, _I32, _VP, _VP, _VP]
    L.mk_get_status.argtypes = [_VP]
    L.mk_set_wait_timeout.argtypes = [_VP, ctypes.c_uint64]
    L.mk_set_trace.argtypes = [_VP, _I32]
    L.mk_set_sampling.argtypes = [_VP, ctypes.c_float, ctypes.c_uint64]
    L.mk_read_trace.argtypes = [_VP, ctypes.POINTER(ctypes.c_int64), _I32]
    L.mk_plan_size.argtypes = [_VP, _PI32, _PI32]
    L.mk_plan_inspect.argtypes = [ctypes.POINTER(mk_config), _I32, _PI32, _I32, _PI32, _PI32]
    L.mk_debug_read.argtypes = [_VP, ctypes.POINTER(ctypes.c_uint64)]
    L.mk_decode_step_noalloc.argtypes = [ctypes.POINTER(mk_config), ctypes.POINTER(mk_weights),
                                         ctypes.POINTER(mk_kv_cache), _I32, _I32, _VP, _VP, _VP]
    L.mk_set_sampling_filter.argtypes = [_VP, _I32, ctypes.c_float]
    L.mk_sampling_noise.argtypes = [_I32, _I32, _I32, ctypes.c_uint64, _VP, _VP, _VP, _VP]
    L.mk_draw_from_logits.argtypes = [_VP, _I32, _I32, ctypes.c_float, _I32, ctypes.c_float, _VP, ctypes.c_uint64,
                                      _VP, _VP]
    L.mk_w2_pack.argtypes = [_VP, ctypes.c_int64, ctypes.c_int64, _VP]
    L.mk_w2_unpack.argtypes = [_VP, ctypes.c_int64, ctypes.c_int64, _VP]
    L.mk_w2a8_gemv.argtypes = [_VP, ctypes.c_float, _I32, _I32, _VP, _VP, _VP]
    L.mk_twell_down.argtypes = [_VP, _I32, _I32, _VP, _VP, _VP]
    L.mk_twell_ffn.argtypes = [_VP, _VP, _VP, _I32, _I32, _VP, _VP, _VP, _VP]
    L.mk_prefill.argtypes = [_VP, _VP, _I32, _I32, _VP, _VP, _VP]
    L.mk_tc_gemm.argtypes = [_VP, _I32, _I32, _VP, _VP, _I32, _VP, _VP, _VP, _VP]
    L.mk_destroy.argtypes = [_VP]
    L.mk_destroy.restype = None
    _lib = L
    return L


def declared_symbols(header: str = HEADER) -> list[str]:
    """Function names declared in include/mk.h."""
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mk_[a-z_0-9]+)\s*\(", text)))


def check(rc: int) -> int:
    if rc < 0:
        raise MKError(rc, load().mk_last_error().decode())
    return rc


def make_config(shape, max_seq: int, max_batch: int = 1, attn_splits: int = 0) -> mk_config:
    return mk_config(shape.n_layers, shape.d_model, shape.n_heads, shape.n_kv_heads,
                     shape.head_dim, shape.ffn_dim, shape.vocab, int(max_seq), int(max_batch),
                     int(attn_splits), float(shape.rms_eps), float(shape.rope_theta))


def plan_inspect(shape, n_sm: int, max_seq: int, attn_splits: int = 0, max_batch: int = 1):
    """Host-only plan: returns (instr int32 [n, 16] as list of lists, queue lengths, n_counters).
    max_batch > 1 gives the fused batched step's plan where the model supports it."""
    import numpy as np
    L = load()
    cfg = make_config(shape, max_seq, max_batch, attn_splits)
    qlen = (ctypes.c_int32 * n_sm)()
    nctr = ctypes.c_int32(0)
    n = check(L.mk_plan_inspect(ctypes.byref(cfg), n_sm, None, 0, qlen, ctypes.byref(nctr)))
    buf = np.zeros((n, MK_INSTR_WORDS), dtype=np.int32)
    check(L.mk_plan_inspect(ctypes.byref(cfg), n_sm,
                            buf.ctypes.data_as(_PI32), n, qlen, ctypes.byref(nctr)))
    return buf, np.array(list(qlen), dtype=np.int64), int(nctr.value)


def _stream_ptr(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _weights_struct(shape, weights: dict):
    layers = (mk_layer_weights * shape.n_layers)()
    for i, lw in enumerate(weights["layers"]):
        for k in ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down"):
            setattr(layers[i], k, lw[k].data_ptr())
    w = mk_weights(weights["embed"].data_ptr(), weights["final_norm"].data_ptr(),
                   ctypes.cast(layers, ctypes.POINTER(mk_layer_weights)))
    return w, layers


def decode_step_noalloc(shape, weights: dict, k_cache, v_cache, token: int, pos: int, out_token,
                        logits=None, attn_splits: int = 0, stream=None) -> None:
    """mk_decode_step_noalloc: one decode step without a handle and without
    any device allocation (scratch lives in the library's static array)."""
    cfg = make_config(shape, int(k_cache.shape[3]), int(k_cache.shape[1]), attn_splits)
    w, layers = _weights_struct(shape, weights)
    kv = mk_kv_cache(k_cache.data_ptr(), v_cache.data_ptr())
    check(load().mk_decode_step_noalloc(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(kv),
                                        int(token), int(pos),
                                        logits.data_ptr() if logits is not None else None,
                                        out_token.data_ptr(), _stream_ptr(stream)))


def sampling_noise(n: int, position: int, slot: int, seed: int, out_words=None, out_noise=None,
                   words=None, stream=None) -> None:
    """mk_sampling_noise: the sampling epilogue's Philox words and Gumbel noise for
    vocabulary entries 0..n-1 (int32/uint32 and float32 CUDA tensors [n]); with
    `words` given, the noise of those words instead."""
    ptr = lambda t: t.data_ptr() if t is not None else None
    check(load().mk_sampling_noise(int(n), int(position), int(slot), int(seed) & ((1 << 64) - 1),
                                   ptr(words), ptr(out_words), ptr(out_noise), _stream_ptr(stream)))


def draw_from_logits(logits, temperature: float, top_k: int, top_p: float, positions, seed: int, out_tokens,
                     stream=None) -> None:
    """mk_draw_from_logits: logits float32 CUDA tensor [B][V]; positions and
    out_tokens int32 CUDA tensors [B]; sequence b draws on slot b's noise."""
    B, V = int(logits.shape[0]), int(logits.shape[1])
    check(load().mk_draw_from_logits(logits.data_ptr(), B, V, float(temperature), int(top_k), float(top_p),
                                     positions.data_ptr(), int(seed) & ((1 << 64) - 1), out_tokens.data_ptr(),
                                     _stream_ptr(stream)))


def w2_pack(q):
    """Host: ternary int8 codes [rows][cols] (numpy) -> packed uint32 [rows][cols / 16]
    in the library's W2 layout (mk_w2_pack)."""
    import numpy as np
    q = np.ascontiguousarray(q, dtype=np.int8)
    rows, cols = q.shape
    out = np.empty((rows, cols // 16), dtype=np.uint32)
    check(load().mk_w2_pack(q.ctypes.data, rows, cols, out.ctypes.data))
    return out


def w2_unpack(packed, cols: int):
    """Host: the inverse of w2_pack (mk_w2_unpack)."""
    import numpy as np
    packed = np.ascontiguousarray(packed, dtype=np.uint32)
    rows = packed.shape[0]
    out = np.empty((rows, cols), dtype=np.int8)
    check(load().mk_w2_unpack(packed.ctypes.data, rows, cols, out.ctypes.data))
    return out


def w2a8_gemv(packed, beta: float, rows: int, cols: int, x, y, stream=None) -> None:
    """mk_w2a8_gemv on CUDA tensors: packed (uint32/int32 [rows][cols/16]),
    x float32 [cols], y float32 [rows]."""
    check(load().mk_w2a8_gemv(packed.data_ptr(), float(beta), int(rows), int(cols), x.data_ptr(),
                              y.data_ptr(), _stream_ptr(stream)))


def twell_down(w_down_t, h, y, stream=None) -> None:
    """mk_twell_down on CUDA tensors: w_down_t bf16 [F][d], h float32 [F],
    y float32 [d] = W_down h over the non-zero entries of h."""
    F, d = w_down_t.shape
    rc = load().mk_twell_down(w_down_t.data_ptr(), int(F), int(d), h.data_ptr(), y.data_ptr(), _stream_ptr(stream))
    if rc != 0:
        raise MKError(rc, f"mk_twell_down returned {rc}")


def twell_ffn(w_gate, w_up, w_down_t, x, h, y, stream=None) -> None:
    """mk_twell_ffn on CUDA tensors: w_gate / w_up bf16 [F][d], w_down_t bf16
    [F][d], x float32 [d]; writes h float32 [F] = relu(W_gate x) * (W_up x) and
    y float32 [d] = W_down h."""
    F, d = w_gate.shape
    rc = load().mk_twell_ffn(w_gate.data_ptr(), w_up.data_ptr(), w_down_t.data_ptr(), int(F), int(d),
                             x.data_ptr(), h.data_ptr(), y.data_ptr(), _stream_ptr(stream))
    if rc != 0:
        raise MKError(rc, f"mk_twell_ffn returned {rc}")


def tc_gemm(w, bhi, blo, y, r=None, status=None, stream=None) -> None:
    """mk_tc_gemm on CUDA tensors: w bf16 [M][K], bhi / blo bf16 [N][K], y (and r)
    float32 [N][M]; y = W (bhi + blo)^T (+ r). status: int32 CUDA tensor [1]
    (zeroed by the caller) that turns non-zero if an in-kernel wait expires;
    without it, the call synchronises and raises on expiry."""
    import torch
    M, K = w.shape
    N = bhi.shape[0]
    st = status if status is not None else torch.zeros(1, dtype=torch.int32, device=y.device)
    rc = load().mk_tc_gemm(w.data_ptr(), int(M), int(K), bhi.data_ptr(), blo.data_ptr(), int(N), y.data_ptr(),
                           r.data_ptr() if r is not None else None, st.data_ptr(), _stream_ptr(stream))
    if rc != 0:
        raise MKError(rc, f"mk_tc_gemm returned {rc}")
    if status is None and int(st.item()) != 0:
        raise MKError(MK_ERR_TIMEOUT, "a bounded wait of the tensor-core contraction expired")


class Megakernel:
    """One model bound to the decode megakernel (owns an mk_handle).

    weights: dict from synth.make_weights on a CUDA device (bf16 tensors).
    k_cache, v_cache: bf16 CUDA tensors [L][max_batch][Hkv][max_seq][hd].
    """

    def __init__(self, shape, weights: dict, k_cache, v_cache, attn_splits: int = 0):
        L = load()
        self.shape = shape
        self.max_seq = int(k_cache.shape[3])
        self.max_batch = int(k_cache.shape[1])
        self._keep = (weights, k_cache, v_cache)
        self.cfg = make_config(shape, self.max_seq, self.max_batch, attn_splits)
        w, layers = _weights_struct(shape, weights)
        self._layers = layers
        kv = mk_kv_cache(k_cache.data_ptr(), v_cache.data_ptr())
        h = _VP()
        check(L.mk_create(ctypes.byref(self.cfg), ctypes.byref(w), ctypes.byref(kv), ctypes.byref(h)))
        self.h = h

    def step(self, token: int, pos: int, out_token, logits=None, stream=None) -> None:
        check(load().mk_decode_step(self.h, int(token), int(pos),
                                    logits.data_ptr() if logits is not None else None,
                                    out_token.data_ptr(), _stream_ptr(stream)))

    def step_dev(self, d_token, pos: int, out_token, logits=None, stream=None) -> None:
        check(load().mk_decode_step_dev(self.h, d_token.data_ptr(), int(pos),
                                        logits.data_ptr() if logits is not None else None,
                                        out_token.data_ptr(), _stream_ptr(stream)))

    def step_batch(self, d_tokens, d_positions, out_tokens, logits=None, stream=None) -> None:
        """d_tokens, d_positions, out_tokens: int32 CUDA tensors [B]; logits: float32 CUDA
        tensor [B][vocab] or None. Sequence b uses batch slot b of the KV cache. With
        B == max_batch (head dim 64) all sequences run in one fused launch that reads
        every weight tile once (fp16 GEMV inputs; with a top-k / top-p filter, two
        short draw kernels follow it); otherwise one launch per sequence."""
        check(load().mk_decode_step_batch(self.h, d_tokens.data_ptr(), d_positions.data_ptr(),
                                          int(d_tokens.numel()),
                                          logits.data_ptr() if logits is not None else None,
                                          out_tokens.data_ptr(), _stream_ptr(stream)))

    def prefill(self, d_tokens, start_pos: int, out_token, logits=None, stream=None) -> None:
        """mk_prefill: d_tokens int32 CUDA tensor [n] at positions start_pos ..;
        out_token int32 CUDA tensor [1]; logits float32 CUDA tensor [vocab] or None."""
        check(load().mk_prefill(self.h, d_tokens.data_ptr(), int(d_tokens.numel()), int(start_pos),
                                logits.data_ptr() if logits is not None else None, out_token.data_ptr(),
                                _stream_ptr(stream)))

    def step_unfused(self, token: int, pos: int, out_token, logits=None, stream=None) -> None:
        check(load().mk_decode_step_unfused(self.h, int(token), int(pos),
                                            logits.data_ptr() if logits is not None else None,
                                            out_token.data_ptr(), _stream_ptr(stream)))

    def step_host(self, host_token, pos: int, host_out_token, host_logits=None, stream=None) -> None:
        """host_token / host_out_token: pinned int32 CPU tensors [1]; host_logits: pinned
        float32 CPU tensor [vocab] or None."""
        check(load().mk_decode_step_host(
            self.h, ctypes.cast(host_token.data_ptr(), _PI32), int(pos),
            host_logits.data_ptr() if host_logits is not None else None,
            ctypes.cast(host_out_token.data_ptr(), _PI32), _stream_ptr(stream)))

    def status(self) -> int:
        return load().mk_get_status(self.h)

    def set_wait_timeout(self, ns: int) -> None:
        check(load().mk_set_wait_timeout(self.h, int(ns)))

    def set_sampling(self, temperature: float, seed: int = 0) -> None:
        """temperature > 0: tokens are drawn from softmax(logits / temperature)
        (Gumbel-max with Philox noise keyed by seed); <= 0: greedy."""
        check(load().mk_set_sampling(self.h, float(temperature), int(seed) & ((1 << 64) - 1)))

    def set_sampling_filter(self, top_k: int = 0, top_p: float = 1.0) -> None:
        """Top-k / top-p filtering of the sampled draw (mk_set_sampling_filter);
        top_k = 0 and top_p = 1 switch it off."""
        check(load().mk_set_sampling_filter(self.h, int(top_k), float(top_p)))

    def set_trace(self, on: bool) -> None:
        check(load().mk_set_trace(self.h, 1 if on else 0))

    def read_trace(self):
        import numpy as np
        need = check(load().mk_read_trace(self.h, None, 0))
        buf = np.zeros((max(1, need), 8), dtype=np.int64)
        n = check(load().mk_read_trace(self.h, buf.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                       buf.shape[0]))
        return buf[:n]

    def debug_read(self):
        """(checked_build, [site, address, bytes, block<<32|thread])."""
        out = (ctypes.c_uint64 * 4)()
        rc = check(load().mk_debug_read(self.h, out))
        return rc == 1, list(out)

    def plan_size(self):
        n_sm, n_instr = ctypes.c_int32(), ctypes.c_int32()
        check(load().mk_plan_size(self.h, ctypes.byref(n_sm), ctypes.byref(n_instr)))
        return n_sm.value, n_instr.value

    def close(self) -> None:
        if getattr(self, "h", None):
            load().mk_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
