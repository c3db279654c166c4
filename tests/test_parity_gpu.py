"""GPU parity: the megakernel (through the C ABI) against the fp64 oracle,
teacher-forced, step by step, on every workload shape; plus the unfused
chain, determinism, device/host entry points, argument checks and the
bounded-wait failure path."""
import numpy as np
import pytest
import torch

from decode_megakernel_llama_gb300 import _lib, synth
from decode_megakernel_llama_gb300.configs import LLAMA_1B, LLAMA_3B, TINY, WORKLOADS, ModelShape

from gpu_helpers import Pair, compare, teacher_forced

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny(cuda_dev):
    wl = WORKLOADS["tiny"]
    p = Pair(TINY, wl.max_seq)
    yield p
    p.close()


def test_tiny_full_workload_teacher_forced(tiny):
    wl = WORKLOADS["tiny"]
    prompt = synth.prompt_tokens(TINY.vocab, wl.prompt_len)
    stats = teacher_forced(tiny, prompt, wl.decode_steps)
    assert len(stats) == wl.prompt_len + wl.decode_steps


def test_tiny_unfused_chain_is_bitwise_equal_to_megakernel(cuda_dev):
    a = Pair(TINY, 16)
    b = Pair(TINY, 16)
    for pos, tok in enumerate([5, 77, 4095, 0, 123]):
        la, ta = a.gpu_step(tok, pos, "mega")
        lb, tb = b.gpu_step(tok, pos, "unfused")
        np.testing.assert_array_equal(la, lb)
        assert ta == tb
    torch.testing.assert_close(a.k, b.k, rtol=0, atol=0)
    a.close()
    b.close()


def test_tiny_deterministic_across_runs(cuda_dev):
    outs = []
    for _ in range(2):
        p = Pair(TINY, 12)
        outs.append([p.gpu_step(t, i)[0] for i, t in enumerate([3, 1, 4, 1, 5, 9])])
        p.close()
    for x, y in zip(*outs):
        np.testing.assert_array_equal(x, y)


def test_multi_tile_multi_split_attention_with_ragged_tail(cuda_dev):
    # 300 pre-filled positions: 128-position tiles, 3 forced splits, a ragged
    # last tile, then a few decode steps crossing no boundary.
    shape = TINY
    p = Pair(shape, 320, prefill=300, attn_splits=3)
    teacher_forced(p, [7], 6, start_pos=300)
    p.close()


@pytest.mark.parametrize("splits", [1, 2, 5])
def test_split_counts_agree(cuda_dev, splits):
    p = Pair(TINY, 400, prefill=385, attn_splits=splits)
    teacher_forced(p, [11, 12], 2, start_pos=385)
    p.close()


def test_head_dim_128_and_group_3(cuda_dev):
    shape = ModelShape("hd128-g3", 2, 768, 6, 2, 128, 1536, 2048, 1e-5, 5e5)
    p = Pair(shape, 200, prefill=130)
    teacher_forced(p, [9, 8], 3, start_pos=130)
    p.close()


def test_vocab_not_a_multiple_of_the_tile(cuda_dev):
    shape = ModelShape("odd-vocab", 1, 256, 4, 4, 64, 512, 1001, 1e-5, 1e4)
    p = Pair(shape, 8)
    teacher_forced(p, [1000, 0, 500], 2)
    p.close()


def test_llama1b_teacher_forced(cuda_dev):
    # the whole workload: 128 prompt tokens and all 128 greedy decode steps
    wl = WORKLOADS["llama1b"]
    p = Pair(LLAMA_1B, wl.max_seq)
    prompt = synth.prompt_tokens(LLAMA_1B.vocab, wl.prompt_len)
    stats = teacher_forced(p, prompt, wl.decode_steps, check_every=8)
    p.close()
    assert len(stats) >= (wl.prompt_len + wl.decode_steps) // 8
    assert max(s[0] for s in stats) <= 5e-2


def test_llama1b_long_context_prefilled_8192(cuda_dev):
    # the whole workload: 8192 cached positions, then 64 decode steps
    wl = WORKLOADS["llama1b_ctx8192"]
    p = Pair(LLAMA_1B, wl.max_seq, prefill=wl.prefill)
    prompt = synth.prompt_tokens(LLAMA_1B.vocab, wl.prompt_len)
    stats = teacher_forced(p, prompt, wl.decode_steps, start_pos=wl.prefill)
    p.close()
    assert len(stats) == wl.prompt_len + wl.decode_steps


def test_llama3b_teacher_forced(cuda_dev):
    # the whole workload: 256 prompt tokens and all 128 greedy decode steps
    # (head dim 128, three query heads per kv head)
    wl = WORKLOADS["llama3b"]
    p = Pair(LLAMA_3B, wl.max_seq)
    prompt = synth.prompt_tokens(LLAMA_3B.vocab, wl.prompt_len)
    stats = teacher_forced(p, prompt, wl.decode_steps, check_every=16)
    p.close()
    assert len(stats) >= (wl.prompt_len + wl.decode_steps) // 16


def test_device_token_chaining_matches_host_token(tiny):
    # the same cache positions are rewritten with identical values
    dev = torch.device("cuda:0")
    d_tok = torch.tensor([42], dtype=torch.int32, device=dev)
    out = torch.zeros(1, dtype=torch.int32, device=dev)
    la = torch.empty(TINY.vocab, device=dev)
    tiny.mk.step(42, 0, out, la)
    torch.cuda.synchronize()
    ref = la.clone()
    tiny.mk.step_dev(d_tok, 0, d_tok, la)   # in-place chaining: token in = token out
    torch.cuda.synchronize()
    assert tiny.mk.status() == 0
    torch.testing.assert_close(la, ref, rtol=0, atol=0)
    assert int(d_tok.item()) == int(out.item())


def test_host_entry_point(tiny):
    ht = torch.tensor([42], dtype=torch.int32).pin_memory()
    ho = torch.zeros(1, dtype=torch.int32).pin_memory()
    hl = torch.empty(TINY.vocab, dtype=torch.float32).pin_memory()
    tiny.mk.step_host(ht, 0, ho, hl)
    gl, gt = tiny.gpu_step(42, 0)
    np.testing.assert_array_equal(hl.double().numpy(), gl)
    assert int(ho.item()) == gt


def test_invalid_arguments_rejected_on_host(tiny):
    out = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    with pytest.raises(_lib.MKError) as e:
        tiny.mk.step(TINY.vocab, 0, out)
    assert e.value.code == _lib.MK_ERR_INVALID_ARG
    with pytest.raises(_lib.MKError):
        tiny.mk.step(0, tiny.max_seq, out)
    with pytest.raises(_lib.MKError):
        tiny.mk.step(-1, 0, out)


def test_device_token_out_of_range_sets_status_and_touches_nothing(tiny):
    dev = torch.device("cuda:0")
    before = tiny.k.clone()
    bad = torch.tensor([TINY.vocab + 5], dtype=torch.int32, device=dev)
    out = torch.full((1,), -7, dtype=torch.int32, device=dev)
    tiny.mk.step_dev(bad, 3, out)
    torch.cuda.synchronize()
    assert tiny.mk.status() == _lib.MK_ERR_INVALID_ARG
    assert int(out.item()) == -7
    torch.testing.assert_close(tiny.k, before, rtol=0, atol=0)
    # the handle works again after the status was read
    gl, gt = tiny.gpu_step(1, 0)
    assert np.isfinite(gl).all()


def test_expired_wait_reports_timeout_and_recovers(cuda_dev):
    # A 1 ns wait limit makes the first dependency wait that is not already
    # satisfied give up: the kernel records MK_ERR_TIMEOUT, drains its copies
    # and returns; the handle then works normally again.
    p = Pair(LLAMA_1B, 64)
    ref_l, ref_t = p.gpu_step(17, 0)
    p.mk.set_wait_timeout(1)
    p.mk.step(17, 0, p.tok, p.logits)
    torch.cuda.synchronize()
    assert p.mk.status() == _lib.MK_ERR_TIMEOUT
    p.mk.set_wait_timeout(2_000_000_000)
    l2, t2 = p.gpu_step(17, 0)
    np.testing.assert_array_equal(l2, ref_l)
    assert t2 == ref_t
    p.close()


def test_trace_records_every_instruction(tiny):
    tiny.mk.set_trace(True)
    tiny.gpu_step(3, 0)
    tr = tiny.mk.read_trace()
    tiny.mk.set_trace(False)
    n_sm, n_instr = tiny.mk.plan_size()
    assert len(tr) == n_instr
    assert set(np.unique(tr[:, 1])) <= {1, 2, 3, 4, 5, 6}
    assert (tr[:, 2] <= tr[:, 3]).all() and (tr[:, 3] <= tr[:, 7]).all()  # tile wait >= 0
    assert ((tr[:, 4] >= tr[:, 3]) & (tr[:, 6] <= tr[:, 7])).all()
