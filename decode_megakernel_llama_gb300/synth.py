"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke
check. Holds none of the decode arithmetic: only random draws, dtype casts
and host copies.

Recipe: every matrix bf16(N(0, 0.02)); norm gains bf16(1 + N(0, 0.05)); drawn
from one torch generator seeded `seed` in the fixed order embed, then per
layer attn_norm, wq, wk, wv, wo, mlp_norm, w_gate, w_up, w_down, then
final_norm. Prompt tokens are uniform in [0, vocab) from a CPU generator
(seed 1, sequence b of a batch: seed 100 + b). Pre-filled cache entries are
bf16(N(0, 1)) from seed 2.
"""
from __future__ import annotations

import numpy as np
import torch

from .configs import ModelShape

LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")


def layer_shapes(s: ModelShape) -> dict:
    d, F = s.d_model, s.ffn_dim
    return {
        "attn_norm": (d,), "wq": (s.q_dim, d), "wk": (s.kv_dim, d), "wv": (s.kv_dim, d),
        "wo": (d, s.q_dim), "mlp_norm": (d,), "w_gate": (F, d), "w_up": (F, d),
        "w_down": (d, F),
    }


def _normal(shape, std, mean, gen, device):
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(torch.bfloat16)


def make_weights(s: ModelShape, device="cpu", seed: int = 0) -> dict:
    """Random-init bf16 weights of shape `s` on `device`."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    w = {"embed": _normal((s.vocab, s.d_model), 0.02, 0.0, gen, device), "layers": []}
    for _ in range(s.n_layers):
        lw = {}
        for k, shp in layer_shapes(s).items():
            if k.endswith("norm"):
                lw[k] = _normal(shp, 0.05, 1.0, gen, device)
            else:
                lw[k] = _normal(shp, 0.02, 0.0, gen, device)
        w["layers"].append(lw)
    w["final_norm"] = _normal((s.d_model,), 0.05, 1.0, gen, device)
    return w


def prompt_tokens(vocab: int, n: int, seq: int = 0) -> torch.Tensor:
    gen = torch.Generator(device="cpu")
    gen.manual_seed(1 if seq == 0 else 100 + seq)
    return torch.randint(0, vocab, (n,), generator=gen, dtype=torch.int64).to(torch.int32)


def kv_cache(s: ModelShape, max_seq: int, batch: int = 1, device="cpu") -> tuple:
    """Zeroed bf16 caches [L][B][Hkv][max_seq][hd]."""
    shape = (s.n_layers, batch, s.n_kv_heads, max_seq, s.head_dim)
    return (torch.zeros(shape, dtype=torch.bfloat16, device=device),
            torch.zeros(shape, dtype=torch.bfloat16, device=device))


def prefill_cache(k: torch.Tensor, v: torch.Tensor, n_positions: int, seed: int = 2) -> None:
    """Fill positions [0, n_positions) of both caches with bf16(N(0,1))."""
    gen = torch.Generator(device=k.device)
    gen.manual_seed(seed)
    shape = k[:, :, :, :n_positions, :].shape
    k[:, :, :, :n_positions, :] = _normal(shape, 1.0, 0.0, gen, k.device)
    v[:, :, :, :n_positions, :] = _normal(shape, 1.0, 0.0, gen, k.device)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Host copy of a bf16 tensor as its raw uint16 bit patterns."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_weights(w: dict) -> dict:
    """The same weights as host uint16 bit arrays (what the oracle reads)."""
    return {
        "embed": bf16_bits(w["embed"]),
        "final_norm": bf16_bits(w["final_norm"]),
        "layers": [{k: bf16_bits(v) for k, v in lw.items()} for lw in w["layers"]],
    }


W2_MATS = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")
W2_BETAS = ("beta_q", "beta_k", "beta_v", "beta_o", "beta_gate", "beta_up", "beta_down")


def make_ternary_weights(s: ModelShape, device="cpu", seed: int = 0) -> dict:
    """A ternary-weight model of shape `s` (the W2A8 variant): embedding and
    norm gains drawn as in make_weights (bf16), every projection matrix a
    uniform draw from {-1, 0, +1} (int8) with one scale per matrix drawn
    uniformly from [0.02, 0.03] and rounded to a bf16 value (so beta * Wq is
    exact in bf16), which gives the matrices about the spread of the bf16
    model's N(0, 0.02) weights. Recipe order: embed, then per layer
    attn_norm, the seven matrices and their scales in W2_MATS order,
    mlp_norm; then final_norm."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    shapes = layer_shapes(s)
    w = {"embed": _normal((s.vocab, s.d_model), 0.02, 0.0, gen, device), "layers": []}
    for _ in range(s.n_layers):
        lw = {"attn_norm": _normal(shapes["attn_norm"], 0.05, 1.0, gen, device)}
        for m, b in zip(W2_MATS, W2_BETAS):
            lw[m] = (torch.randint(0, 3, shapes[m], generator=gen, device=device, dtype=torch.int32) - 1).to(torch.int8)
            u = torch.rand((1,), generator=gen, device=device, dtype=torch.float32)
            lw[b] = float((0.02 + 0.01 * u).to(torch.bfloat16).float().item())
        lw["mlp_norm"] = _normal(shapes["mlp_norm"], 0.05, 1.0, gen, device)
        w["layers"].append(lw)
    w["final_norm"] = _normal((s.d_model,), 0.05, 1.0, gen, device)
    return w


def host_ternary_weights(w: dict) -> dict:
    """The ternary model on the host: bf16 bits, int8 codes, float scales."""
    out = {"embed": bf16_bits(w["embed"]), "final_norm": bf16_bits(w["final_norm"]), "layers": []}
    for lw in w["layers"]:
        h = {k: bf16_bits(lw[k]) for k in ("attn_norm", "mlp_norm")}
        for m, b in zip(W2_MATS, W2_BETAS):
            h[m] = lw[m].detach().contiguous().cpu().numpy()
            h[b] = lw[b]
        out["layers"].append(h)
    return out


def sparse_activations(F: int, sparsity: float, seed: int = 5, device="cpu") -> torch.Tensor:
    """float32 [F]: exactly round(sparsity * F) zeros at seeded random places,
    the other entries N(0, 1) (a stand-in for the hidden activations of a
    ReLU-gated FFN block of a trained model, whose sparsity random weights do
    not reproduce)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    h = torch.randn(F, generator=g, dtype=torch.float32)
    nz = int(round(sparsity * F))
    if nz > 0:
        h[torch.randperm(F, generator=g)[:nz]] = 0.0
    return h.to(device)
