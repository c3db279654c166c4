"""GPU parity of the batched entry point (mk_decode_step_batch): each
sequence of the batch against its own oracle twin, teacher-forced, with
device-resident tokens and positions and one KV-cache slot per sequence."""
import os

import numpy as np
import pytest
import torch

import oracle
from decode_megakernel_llama_gb300 import _lib, synth
from decode_megakernel_llama_gb300.build import build
from decode_megakernel_llama_gb300.configs import LLAMA_1B, TINY, WORKLOADS, ModelShape

from gpu_helpers import MARGIN, MAX_ABS, compare, oracle_config

pytestmark = pytest.mark.gpu


class BatchPair:
    """The batched entry point on cuda:0 and one oracle per sequence. With
    `prefill`, cache positions [0, prefill) of every slot hold seeded
    bf16(N(0,1)) keys and values (the stand-in for prompts run in lockstep),
    copied byte for byte into each sequence's oracle cache."""

    def __init__(self, shape, max_seq: int, batch: int, prefill: int = 0, attn_splits: int = 0):
        build()
        oracle.set_threads(os.cpu_count() or 1)
        dev = torch.device("cuda:0")
        self.shape, self.B = shape, batch
        self.w = synth.make_weights(shape, dev, 0)
        self.k, self.v = synth.kv_cache(shape, max_seq, batch, dev)
        if prefill:
            synth.prefill_cache(self.k, self.v, prefill)
        self.mk = _lib.Megakernel(shape, self.w, self.k, self.v, attn_splits=attn_splits)
        hw = synth.host_weights(self.w)
        self.orc = [oracle.OracleModel(oracle_config(shape), hw, max_seq) for _ in range(batch)]
        if prefill:
            for b in range(batch):
                self.orc[b].k_cache[:] = synth.bf16_bits(self.k[:, b])
                self.orc[b].v_cache[:] = synth.bf16_bits(self.v[:, b])
        self.tok_in = torch.zeros(batch, dtype=torch.int32, device=dev)
        self.pos_in = torch.zeros(batch, dtype=torch.int32, device=dev)
        self.tok_out = torch.zeros(batch, dtype=torch.int32, device=dev)
        self.logits = torch.empty(batch, shape.vocab, dtype=torch.float32, device=dev)

    def step(self, tokens, positions):
        self.tok_in.copy_(torch.tensor(tokens, dtype=torch.int32))
        self.pos_in.copy_(torch.tensor(positions, dtype=torch.int32))
        self.mk.step_batch(self.tok_in, self.pos_in, self.tok_out, self.logits)
        torch.cuda.synchronize()
        assert self.mk.status() == 0, _lib.load().mk_last_error()
        return self.logits.double().cpu().numpy(), self.tok_out.cpu().numpy().tolist()

    def close(self):
        self.mk.close()


def run_lockstep(bp: BatchPair, prompts, n_decode: int, check_from: int = 0, start_pos: int = 0):
    """Teacher-forced lockstep: every sequence gets its prompt, then its own
    oracle's greedy tokens; all sequences sit at the same position."""
    nxt = [None] * bp.B
    n = len(prompts[0])
    worst = 0.0
    for i in range(n + n_decode):
        toks = [int(prompts[b][i]) if i < n else nxt[b] for b in range(bp.B)]
        pos = start_pos + i
        gl, gt = bp.step(toks, [pos] * bp.B)
        for b in range(bp.B):
            ol, ot = bp.orc[b].decode_step(toks[b], pos)
            if i >= check_from:
                worst = max(worst, compare(gl[b], gt[b], ol, ot, f"seq {b} step {i} pos {pos}")[0])
            nxt[b] = ot
    return worst


def test_tiny_batch3_lockstep_teacher_forced(cuda_dev):
    bp = BatchPair(TINY, 24, 3)
    prompts = [synth.prompt_tokens(TINY.vocab, 6, seq=b) for b in range(3)]
    run_lockstep(bp, prompts, 10)
    bp.close()


def test_tiny_batch_positions_differ_per_sequence(cuda_dev):
    # sequence 0 runs two steps ahead through the single-sequence call (slot 0),
    # then both advance together at different positions
    bp = BatchPair(TINY, 24, 2)
    torch_tok = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    lg = torch.empty(TINY.vocab, dtype=torch.float32, device="cuda:0")
    for pos, tok in enumerate([17, 230]):
        bp.mk.step(tok, pos, torch_tok, lg)
        bp.orc[0].decode_step(tok, pos)
    torch.cuda.synchronize()
    toks = [[5, 6, 7], [900, 901, 902]]
    for i in range(3):
        gl, gt = bp.step([toks[0][i], toks[1][i]], [2 + i, i])
        ol0, ot0 = bp.orc[0].decode_step(toks[0][i], 2 + i)
        ol1, ot1 = bp.orc[1].decode_step(toks[1][i], i)
        compare(gl[0], gt[0], ol0, ot0, f"seq 0 step {i}")
        compare(gl[1], gt[1], ol1, ot1, f"seq 1 step {i}")
    bp.close()


def test_batched_step_matches_single_sequence_steps(cuda_dev):
    # the fused batched step (all sequences in one launch) against the same
    # sequences stepped one by one through the single-sequence call: the
    # fused step rounds its GEMV inputs for the tensor cores, the
    # single-sequence step keeps them in fp32, so they agree to the parity
    # tolerance, with the same greedy token wherever the top two logits are
    # clearly apart
    a = BatchPair(TINY, 16, 2)
    singles = [BatchPair(TINY, 16, 1), BatchPair(TINY, 16, 1)]
    out = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    lg = torch.empty(TINY.vocab, dtype=torch.float32, device="cuda:0")
    for pos, toks in enumerate([(3, 9), (1, 2), (4, 7), (1, 1), (5, 0)]):
        la, ta = a.step(list(toks), [pos, pos])
        for b in range(2):
            singles[b].mk.step(toks[b], pos, out, lg)
            torch.cuda.synchronize()
            ls = lg.double().cpu().numpy()
            assert np.abs(la[b] - ls).max() <= MAX_ABS, (pos, b, np.abs(la[b] - ls).max())
            assert ta[b] == int(out.item()) or np.sort(ls)[-1] - np.sort(ls)[-2] < MARGIN
    a.close()
    for s_ in singles:
        s_.close()


def test_device_position_out_of_range_sets_status(cuda_dev):
    bp = BatchPair(TINY, 8, 2)
    bp.tok_in.copy_(torch.tensor([1, 2], dtype=torch.int32))
    bp.pos_in.copy_(torch.tensor([0, 8], dtype=torch.int32))  # 8 == max_seq
    bp.mk.step_batch(bp.tok_in, bp.pos_in, bp.tok_out, bp.logits)
    torch.cuda.synchronize()
    assert bp.mk.status() == _lib.MK_ERR_INVALID_ARG
    with pytest.raises(_lib.MKError):
        bp.mk.step_batch(bp.tok_in[:0], bp.pos_in[:0], bp.tok_out, bp.logits)  # batch 0
    bp.close()


def test_llama1b_batch8_short_lockstep(cuda_dev):
    # the batch-8 workload's shape, on short prompts so the oracle keeps up
    bp = BatchPair(LLAMA_1B, 8, 8)
    prompts = [synth.prompt_tokens(LLAMA_1B.vocab, 3, seq=b) for b in range(8)]
    run_lockstep(bp, prompts, 1, check_from=2)
    bp.close()


def test_wide_vocab_batch2(cuda_dev):
    # a 160000-row vocabulary: 1250 row tiles of the LM head's tensor-core
    # contraction, and 157 slices per sequence for the token draw
    wide = ModelShape("wide-vocab", 2, 256, 4, 2, 64, 1024, 160000, 1e-5, 1e4)
    bp = BatchPair(wide, 8, 2)
    prompts = [synth.prompt_tokens(wide.vocab, 3, seq=b) for b in range(2)]
    run_lockstep(bp, prompts, 2)
    bp.close()


def test_llama1b_batch8_workload_at_its_512_context(cuda_dev):
    # The batch-8 workload as benchmarked: 8 sequences whose caches hold 512
    # seeded positions, then all 64 decode steps in lockstep (positions
    # 512..575). From position 513 on every (sequence, kv head) runs two KV
    # splits of two or more 128-position tiles and merges them across SMs.
    wl = WORKLOADS["llama1b_b8"]
    P = wl.prompt_len
    bp = BatchPair(LLAMA_1B, P + wl.decode_steps + 1, wl.batch, prefill=P)
    instr, _, _ = _lib.plan_inspect(LLAMA_1B, 152, P + wl.decode_steps + 1, max_batch=wl.batch)
    attn = instr[instr[:, 0] == 2]
    assert attn[:, 3].max() == 1  # split index 1 exists: two splits per (sequence, kv head)
    first = [[int(synth.prompt_tokens(LLAMA_1B.vocab, 1, seq=b)[0])] for b in range(wl.batch)]
    worst = run_lockstep(bp, first, wl.decode_steps - 1, start_pos=P)
    assert worst <= MAX_ABS
    bp.close()


def test_tiny_batch4_three_splits_and_a_ragged_tile(cuda_dev):
    # 1100 cached positions: three KV splits of 367 positions each (tiles of
    # 128, 128 and a ragged 111) per (sequence, kv head), merged across SMs
    bp = BatchPair(TINY, 1200, 4, prefill=1100)
    instr, _, _ = _lib.plan_inspect(TINY, 152, 1200, max_batch=4)
    assert instr[instr[:, 0] == 2][:, 3].max() == 2
    prompts = [synth.prompt_tokens(TINY.vocab, 2, seq=b) for b in range(4)]
    run_lockstep(bp, prompts, 4, start_pos=1100)
    bp.close()


def test_weights_beyond_fp16_range_keep_sequence_by_sequence_batches(cuda_dev):
    # One weight beyond fp16's largest finite value (65504) would become an
    # infinity in the batched step's fp16 copy, so the handle runs batches
    # one sequence at a time: bit for bit the single-sequence step.
    build()
    dev = torch.device("cuda:0")
    w = synth.make_weights(TINY, dev, 0)
    w["layers"][1]["w_up"][3, 5] = 70000.0
    k2, v2 = synth.kv_cache(TINY, 8, 2, dev)
    k1, v1 = synth.kv_cache(TINY, 8, 1, dev)
    batched = _lib.Megakernel(TINY, w, k2, v2)
    single = _lib.Megakernel(TINY, w, k1, v1)
    toks = torch.tensor([7, 7], dtype=torch.int32, device=dev)
    pos = torch.zeros(2, dtype=torch.int32, device=dev)
    out = torch.zeros(2, dtype=torch.int32, device=dev)
    lb = torch.empty(2, TINY.vocab, device=dev)
    o1 = torch.zeros(1, dtype=torch.int32, device=dev)
    l1 = torch.empty(TINY.vocab, device=dev)
    for step, tok in enumerate([7, 8, 9]):
        toks.fill_(tok)
        pos.fill_(step)
        batched.step_batch(toks, pos, out, lb)
        single.step(tok, step, o1, l1)
        torch.cuda.synchronize()
        assert batched.status() == 0 and single.status() == 0
        assert torch.isfinite(lb).all()
        torch.testing.assert_close(lb[0], l1, rtol=0, atol=0)
        torch.testing.assert_close(lb[1], l1, rtol=0, atol=0)
    batched.close()
    single.close()
