"""fp64 CPU oracle of one batch-1 Llama-style decode step (ctypes wrapper).

TEST INFRASTRUCTURE ONLY. The test suite, the package smoke check and the
benchmark's CPU-baseline leg are the only users; the product path never
imports this package. The C code shares nothing with the CUDA library.

What it computes follows the article "Revolution der KI-Beschleunigung: Wie
ein Low-Latency Megakernel den Llama-1B Turbo zündet" (dasgeld.co): a bf16
Llama-1B decode forward pass at batch 1 whose fused implementation changes no
result. The step-by-step definition is in oracle.h.

Every function is pinned by tests/test_oracle_pins.py (closed forms,
invariants, numpy float64 library routines, a separately coded full causal
forward). End-to-end logits of random models have no printed values on the
pages: beyond its pinned parts the end-to-end result is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (-O2, OpenMP, no FP contraction)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))):
        return _LIB
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


class _Config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("d_model", ctypes.c_int32),
                ("n_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("ffn_dim", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("rms_eps", ctypes.c_double),
                ("rope_theta", ctypes.c_double)]


_P16 = ctypes.POINTER(ctypes.c_uint16)
_PD = ctypes.POINTER(ctypes.c_double)


class _Layer(ctypes.Structure):
    _fields_ = [(n, _P16) for n in ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm",
                                    "w_gate", "w_up", "w_down")]


class _Weights(ctypes.Structure):
    _fields_ = [("embed", _P16), ("final_norm", _P16), ("layers", ctypes.POINTER(_Layer))]


_P8 = ctypes.POINTER(ctypes.c_int8)


class _LayerW2(ctypes.Structure):
    _fields_ = ([("attn_norm", _P16), ("mlp_norm", _P16)]
                + [(n, _P8) for n in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")]
                + [(n, ctypes.c_float) for n in ("beta_q", "beta_k", "beta_v", "beta_o", "beta_gate",
                                                 "beta_up", "beta_down")])


class _WeightsW2(ctypes.Structure):
    _fields_ = [("embed", _P16), ("final_norm", _P16), ("layers", ctypes.POINTER(_LayerW2))]


class _KV(ctypes.Structure):
    _fields_ = [("k", _P16), ("v", _P16), ("layer_stride", ctypes.c_int64),
                ("max_seq", ctypes.c_int32)]


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        L.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_f64.restype = ctypes.c_double
        L.orc_f64_to_bf16.argtypes = [ctypes.c_double]
        L.orc_f64_to_bf16.restype = ctypes.c_uint16
        L.orc_set_threads.argtypes = [ctypes.c_int]
        L.orc_get_threads.restype = ctypes.c_int
        L.orc_rmsnorm.argtypes = [_PD, _P16, ctypes.c_int, ctypes.c_double, _PD]
        L.orc_matvec.argtypes = [_P16, ctypes.c_int64, ctypes.c_int64, _PD, _PD]
        L.orc_rope.argtypes = [_PD, ctypes.c_int, ctypes.c_int64, ctypes.c_double]
        L.orc_silu.argtypes = [ctypes.c_double]
        L.orc_silu.restype = ctypes.c_double
        L.orc_softmax.argtypes = [_PD, ctypes.c_int, _PD]
        L.orc_attend.argtypes = [_PD, _P16, _P16, ctypes.c_int, ctypes.c_int, _PD]
        L.orc_argmax.argtypes = [_PD, ctypes.c_int]
        L.orc_argmax.restype = ctypes.c_int
        L.orc_decode_step.argtypes = [ctypes.POINTER(_Config), ctypes.POINTER(_Weights),
                                      ctypes.POINTER(_KV), ctypes.c_int, ctypes.c_int, _PD]
        L.orc_decode_step.restype = ctypes.c_int
        L.orc_full_forward.argtypes = [ctypes.POINTER(_Config), ctypes.POINTER(_Weights),
                                       ctypes.POINTER(ctypes.c_int), ctypes.c_int, _PD]
        L.orc_full_forward.restype = ctypes.c_int
        L.orc_w2a8_quantize.argtypes = [_PD, ctypes.c_int, ctypes.POINTER(ctypes.c_int8)]
        L.orc_w2a8_quantize.restype = ctypes.c_float
        L.orc_matvec_w2a8.argtypes = [ctypes.POINTER(ctypes.c_int8), ctypes.c_float, ctypes.c_int64,
                                      ctypes.c_int64, _PD, _PD]
        L.orc_decode_step_w2a8.argtypes = [ctypes.POINTER(_Config), ctypes.POINTER(_WeightsW2),
                                           ctypes.POINTER(_KV), ctypes.c_int, ctypes.c_int, _PD]
        L.orc_decode_step_w2a8.restype = ctypes.c_int
        _lib = L
    return _lib


# ---- array helpers --------------------------------------------------------

def _u16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bits as uint16, got {a.dtype}")
    return a


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p16(a: np.ndarray):
    return a.ctypes.data_as(_P16)


def _pd(a: np.ndarray):
    return a.ctypes.data_as(_PD)


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def get_threads() -> int:
    return int(lib().orc_get_threads())


# ---- primitives -------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    b = _u16(np.asarray(bits, dtype=np.uint16)).ravel()
    f = lib().orc_bf16_to_f64
    return np.array([f(int(v)) for v in b], dtype=np.float64).reshape(np.shape(bits))


def f64_to_bf16(x) -> np.ndarray:
    x = _f64(x)
    f = lib().orc_f64_to_bf16
    return np.array([f(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


def rmsnorm(x, g: np.ndarray, eps: float) -> np.ndarray:
    x = _f64(x)
    g = _u16(g)
    out = np.empty_like(x)
    lib().orc_rmsnorm(_pd(x), _p16(g), x.size, float(eps), _pd(out))
    return out


def matvec(W: np.ndarray, x) -> np.ndarray:
    W = _u16(W)
    x = _f64(x)
    rows, cols = W.shape
    y = np.empty(rows, dtype=np.float64)
    lib().orc_matvec(_p16(W), rows, cols, _pd(x), _pd(y))
    return y


def rope(v, pos: int, theta: float) -> np.ndarray:
    v = _f64(v).copy()
    lib().orc_rope(_pd(v), v.size, int(pos), float(theta))
    return v


def silu(z: float) -> float:
    return float(lib().orc_silu(float(z)))


def softmax(s) -> np.ndarray:
    s = _f64(s)
    p = np.empty_like(s)
    lib().orc_softmax(_pd(s), s.size, _pd(p))
    return p


def attend(q, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    q = _f64(q)
    K = _u16(K)
    V = _u16(V)
    T, hd = K.shape
    o = np.empty(hd, dtype=np.float64)
    lib().orc_attend(_pd(q), _p16(K), _p16(V), T, hd, _pd(o))
    return o


def argmax(v) -> int:
    v = _f64(v)
    return int(lib().orc_argmax(_pd(v), v.size))


# ---- model ----------------------------------------------------------------

@dataclass
class OracleConfig:
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    rms_eps: float = 1e-5
    rope_theta: float = 1e4


_LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")


class OracleModel:
    """A model whose weights are host bf16 bit arrays (numpy uint16).

    `weights` is a dict: "embed" [V,d], "final_norm" [d], "layers" a list of
    dicts with the keys of _LAYER_KEYS, matrices row-major [out, in].
    The KV cache is owned here: k, v uint16 arrays [L][Hkv][max_seq][hd].
    """

    def __init__(self, cfg: OracleConfig, weights: dict, max_seq: int):
        self.cfg = cfg
        self.max_seq = int(max_seq)
        self._keep = []
        self._w = _Weights()
        emb = _u16(weights["embed"])
        fn = _u16(weights["final_norm"])
        self._keep += [emb, fn]
        self._w.embed = _p16(emb)
        self._w.final_norm = _p16(fn)
        layers = (_Layer * cfg.n_layers)()
        for i, lw in enumerate(weights["layers"]):
            for k in _LAYER_KEYS:
                a = _u16(lw[k])
                self._keep.append(a)
                setattr(layers[i], k, _p16(a))
        self._layers = layers
        self._w.layers = ctypes.cast(layers, ctypes.POINTER(_Layer))
        self._c = _Config(cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim,
                          cfg.ffn_dim, cfg.vocab, cfg.rms_eps, cfg.rope_theta)
        shape = (cfg.n_layers, cfg.n_kv_heads, self.max_seq, cfg.head_dim)
        self.k_cache = np.zeros(shape, dtype=np.uint16)
        self.v_cache = np.zeros(shape, dtype=np.uint16)

    def _kv(self) -> _KV:
        kv = _KV()
        kv.k = _p16(self.k_cache)
        kv.v = _p16(self.v_cache)
        kv.layer_stride = self.cfg.n_kv_heads * self.max_seq * self.cfg.head_dim
        kv.max_seq = self.max_seq
        return kv

    def decode_step(self, token: int, pos: int):
        """Returns (logits float64 [V], greedy token)."""
        logits = np.empty(self.cfg.vocab, dtype=np.float64)
        kv = self._kv()
        tok = lib().orc_decode_step(ctypes.byref(self._c), ctypes.byref(self._w), ctypes.byref(kv),
                                    int(token), int(pos), _pd(logits))
        if tok < 0:
            raise ValueError("orc_decode_step rejected its arguments")
        return logits, int(tok)

    def full_forward(self, tokens) -> tuple[np.ndarray, int]:
        toks = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        logits = np.empty(self.cfg.vocab, dtype=np.float64)
        tok = lib().orc_full_forward(ctypes.byref(self._c), ctypes.byref(self._w),
                                     toks.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                                     toks.size, _pd(logits))
        if tok < 0:
            raise ValueError("orc_full_forward rejected its arguments")
        return logits, int(tok)


# ---- W2A8 projections (ternary weights, 8-bit activations) -------------------

W2_MATS = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")
W2_BETAS = ("beta_q", "beta_k", "beta_v", "beta_o", "beta_gate", "beta_up", "beta_down")


def _i8(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.int8:
        raise TypeError(f"expected int8 ternary codes, got {a.dtype}")
    return a


def w2a8_quantize(x) -> tuple[np.ndarray, float]:
    """Per-token absmax 8-bit codes of x and the scale s (fp32 arithmetic)."""
    x = _f64(x)
    q = np.empty(x.size, dtype=np.int8)
    s = lib().orc_w2a8_quantize(_pd(x), x.size, q.ctypes.data_as(_P8))
    return q, float(s)


def matvec_w2a8(Wq: np.ndarray, beta: float, x) -> np.ndarray:
    """y = beta / s * Wq x_q (Wq int8 ternary [rows][cols])."""
    Wq = _i8(Wq)
    x = _f64(x)
    rows, cols = Wq.shape
    y = np.empty(rows, dtype=np.float64)
    lib().orc_matvec_w2a8(Wq.ctypes.data_as(_P8), float(beta), rows, cols, _pd(x), _pd(y))
    return y


class OracleModelW2A8(OracleModel):
    """OracleModel whose projections are W2A8. `weights`: "embed" and
    "final_norm" bf16 bits; "layers" dicts with bf16 "attn_norm",
    "mlp_norm", int8 ternary matrices W2_MATS and float scales W2_BETAS."""

    def __init__(self, cfg: OracleConfig, weights: dict, max_seq: int):
        self.cfg = cfg
        self.max_seq = int(max_seq)
        self._keep = []
        self._ww = _WeightsW2()
        emb, fn = _u16(weights["embed"]), _u16(weights["final_norm"])
        self._keep += [emb, fn]
        self._ww.embed, self._ww.final_norm = _p16(emb), _p16(fn)
        layers = (_LayerW2 * cfg.n_layers)()
        for i, lw in enumerate(weights["layers"]):
            for k in ("attn_norm", "mlp_norm"):
                a = _u16(lw[k])
                self._keep.append(a)
                setattr(layers[i], k, _p16(a))
            for k in W2_MATS:
                a = _i8(lw[k])
                self._keep.append(a)
                setattr(layers[i], k, a.ctypes.data_as(_P8))
            for k in W2_BETAS:
                setattr(layers[i], k, float(lw[k]))
        self._layers = layers
        self._ww.layers = ctypes.cast(layers, ctypes.POINTER(_LayerW2))
        self._c = _Config(cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim,
                          cfg.ffn_dim, cfg.vocab, cfg.rms_eps, cfg.rope_theta)
        shape = (cfg.n_layers, cfg.n_kv_heads, self.max_seq, cfg.head_dim)
        self.k_cache = np.zeros(shape, dtype=np.uint16)
        self.v_cache = np.zeros(shape, dtype=np.uint16)

    def decode_step(self, token: int, pos: int):
        logits = np.empty(self.cfg.vocab, dtype=np.float64)
        kv = self._kv()
        tok = lib().orc_decode_step_w2a8(ctypes.byref(self._c), ctypes.byref(self._ww), ctypes.byref(kv),
                                         int(token), int(pos), _pd(logits))
        if tok < 0:
            raise ValueError("orc_decode_step_w2a8 rejected its arguments")
        return logits, int(tok)

    def full_forward(self, tokens):
        raise NotImplementedError("the W2A8 oracle steps incrementally only")


# ---- activation-sparse FFN ------------------------------------------------
# The TwELL article (iaexpertos.net, "Sakana AI und NVIDIA: TwELL beschleunigt
# LLMs um bis zu 21,9 %"), sections "Die Herausforderung der von GPUs
# ignorierten Sparsity" and the list of what TwELL involves: after a ReLU-type
# activation most hidden units of an FFN block are exactly zero for a given
# token, and kernels that process only the non-zero elements skip the work of
# the zeros without changing the model. The oracle is the dense definition;
# zero terms add nothing to it, so a kernel that skips them reaches the same
# sum up to rounding order.

def relu_glu(Wg: np.ndarray, Wu: np.ndarray, x) -> np.ndarray:
    """Hidden activations of a ReLU-gated FFN: h = max(Wg x, 0) * (Wu x)
    (Wg, Wu bf16 bits [F][d], x float64 [d]); h_i is exactly 0 where the gate
    is <= 0."""
    g = matvec(Wg, x)
    u = matvec(Wu, x)
    return np.where(g > 0.0, g, 0.0) * u


def down_projection(Wd: np.ndarray, h) -> np.ndarray:
    """y = Wd h for Wd bf16 bits [d][F] (the layout of the model's down
    projection) and h float64 [F]."""
    return matvec(Wd, h)
