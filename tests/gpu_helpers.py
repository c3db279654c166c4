"""Shared helpers of the GPU parity tests: build a seeded model on the GPU,
its oracle twin on the host, and run both teacher-forced."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
from decode_megakernel_llama_gb300 import _lib, synth
from decode_megakernel_llama_gb300.build import build

# Tolerances of the parity bar: per step max |dlogit| <= 5e-2, cosine >= 0.9999,
# exact greedy token wherever the oracle's top-2 margin exceeds 0.1.
MAX_ABS = 5e-2
MIN_COS = 0.9999
MARGIN = 0.1


def oracle_config(shape) -> oracle.OracleConfig:
    return oracle.OracleConfig(shape.n_layers, shape.d_model, shape.n_heads, shape.n_kv_heads,
                               shape.head_dim, shape.ffn_dim, shape.vocab, shape.rms_eps,
                               shape.rope_theta)


class Pair:
    """A megakernel model on cuda:0 and the oracle on the same bf16 bytes."""

    def __init__(self, shape, max_seq: int, prefill: int = 0, attn_splits: int = 0, seed: int = 0):
        build()
        oracle.set_threads(os.cpu_count() or 1)
        self.shape = shape
        self.max_seq = max_seq
        dev = torch.device("cuda:0")
        self.w = synth.make_weights(shape, dev, seed)
        self.k, self.v = synth.kv_cache(shape, max_seq, 1, dev)
        if prefill:
            synth.prefill_cache(self.k, self.v, prefill)
        self.mk = _lib.Megakernel(shape, self.w, self.k, self.v, attn_splits=attn_splits)
        self.orc = oracle.OracleModel(oracle_config(shape), synth.host_weights(self.w), max_seq)
        if prefill:
            self.orc.k_cache[:] = synth.bf16_bits(self.k[:, 0])
            self.orc.v_cache[:] = synth.bf16_bits(self.v[:, 0])
        self.logits = torch.empty(shape.vocab, dtype=torch.float32, device=dev)
        self.tok = torch.zeros(1, dtype=torch.int32, device=dev)

    def gpu_step(self, token: int, pos: int, mode: str = "mega"):
        if mode == "mega":
            self.mk.step(token, pos, self.tok, self.logits)
        elif mode == "unfused":
            self.mk.step_unfused(token, pos, self.tok, self.logits)
        else:
            raise ValueError(mode)
        torch.cuda.synchronize()
        st = self.mk.status()
        assert st == 0, f"device status {st}: {_lib.load().mk_last_error()}"
        return self.logits.double().cpu().numpy(), int(self.tok.item())

    def close(self):
        self.mk.close()


def compare(gpu_logits: np.ndarray, gpu_tok: int, orc_logits: np.ndarray, orc_tok: int, where=""):
    d = np.abs(gpu_logits - orc_logits)
    cos = float(gpu_logits @ orc_logits / (np.linalg.norm(gpu_logits) * np.linalg.norm(orc_logits)))
    assert np.isfinite(gpu_logits).all(), where
    assert d.max() <= MAX_ABS, f"{where}: max |dlogit| {d.max():.3e}"
    assert cos >= MIN_COS, f"{where}: cosine {cos:.7f}"
    top2 = np.sort(orc_logits)[-2:]
    if top2[1] - top2[0] > MARGIN:
        assert gpu_tok == orc_tok, f"{where}: token {gpu_tok} != oracle {orc_tok}"
    # the GPU's own argmax must be the argmax of its own logits (lowest index)
    assert gpu_tok == int(np.argmax(gpu_logits)), where
    return float(d.max()), cos


def teacher_forced(pair: Pair, prompt, n_decode: int, start_pos: int = 0, check_every: int = 1,
                   mode: str = "mega"):
    """Feeds the prompt then the oracle's greedy tokens to both sides; returns stats."""
    stats = []
    toks = [int(t) for t in prompt]
    pos = start_pos
    i = 0
    while i < len(toks) + n_decode:
        tok = toks[i] if i < len(toks) else nxt
        ol, ot = pair.orc.decode_step(tok, pos)
        gl, gt = pair.gpu_step(tok, pos, mode)
        if i % check_every == 0 or i == len(toks) + n_decode - 1:
            stats.append(compare(gl, gt, ol, ot, f"step {i} pos {pos}"))
        nxt = ot
        pos += 1
        i += 1
    return stats
