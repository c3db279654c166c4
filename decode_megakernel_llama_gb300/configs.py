"""Model shapes and decode workloads.

The model shapes are Llama-style decoders (pre-norm RMSNorm, rotary
embedding, grouped-query attention, SwiGLU MLP, tied embedding). The
"Llama-1B" shape is the model the megakernel article ("Revolution der
KI-Beschleunigung: Wie ein Low-Latency Megakernel den Llama-1B Turbo zündet",
dasgeld.co) runs at batch 1 in bf16; the other shapes are the small, long
context, 3B-class and batch-8 workloads used to check and measure it.
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class ModelShape:
    name: str
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    rms_eps: float = 1e-5
    rope_theta: float = 1e4

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def weight_elems_per_layer(self) -> int:
        d, F = self.d_model, self.ffn_dim
        return (d * self.q_dim + 2 * d * self.kv_dim + self.q_dim * d + 3 * d * F + 2 * d)

    def step_weight_bytes(self) -> int:
        """bf16 bytes one decode step must read from the weights: every layer
        matrix and norm gain, the final gain, the whole tied embedding for the
        LM head (the embedding-row gather is counted once more)."""
        elems = (self.n_layers * self.weight_elems_per_layer() + self.d_model
                 + self.vocab * self.d_model + self.d_model)
        return 2 * elems

    def kv_read_bytes(self, n_positions: int, batch: int = 1) -> int:
        """bf16 bytes of keys and values attended over (all layers)."""
        return 2 * 2 * self.n_layers * self.kv_dim * n_positions * batch


@dataclass(frozen=True)
class Workload:
    name: str
    shape: ModelShape
    batch: int
    prompt_len: int      # prompt tokens run through the decode step
    decode_steps: int    # greedy steps after the prompt
    prefill: int = 0     # cache positions pre-filled with N(0,1) keys/values

    @property
    def max_seq(self) -> int:
        return self.prefill + self.prompt_len + self.decode_steps


TINY = ModelShape("tiny", 2, 256, 4, 2, 64, 1024, 4096, 1e-5, 1e4)
LLAMA_1B = ModelShape("llama-1b", 16, 2048, 32, 8, 64, 8192, 128256, 1e-5, 5e5)
LLAMA_3B = ModelShape("llama-3b-class", 28, 3072, 24, 8, 128, 8192, 128256, 1e-5, 5e5)

WORKLOADS = {
    "tiny": Workload("tiny", TINY, 1, 8, 32),
    "llama1b": Workload("llama1b", LLAMA_1B, 1, 128, 128),
    "llama1b_ctx8192": Workload("llama1b_ctx8192", LLAMA_1B, 1, 1, 63, prefill=8192),
    "llama3b": Workload("llama3b", LLAMA_3B, 1, 256, 128),
    "llama1b_b8": Workload("llama1b_b8", LLAMA_1B, 8, 512, 64),
}


def shrink(w: Workload, **kw) -> Workload:
    return replace(w, **kw)
