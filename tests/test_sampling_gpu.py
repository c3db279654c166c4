"""GPU parity of the sampling epilogue (mk_set_sampling): the sampled token of
every step against the oracle's Gumbel-max draw on its own fp64 logits with
the same (seed, position, slot) noise, teacher-forced. The token must match
wherever the oracle's top two scores z_i = logit_i / T + g_i are more than
SCORE_MARGIN apart (the logits may differ by the parity tolerance, scaled
by 1/T), and must always be the argmax of the GPU's own logits plus the
oracle's noise."""
import numpy as np
import pytest
import torch

import oracle
from oracle import sampling
from decode_megakernel_llama_gb300 import _lib, synth
from decode_megakernel_llama_gb300.build import build
from decode_megakernel_llama_gb300.configs import LLAMA_1B, TINY, ModelShape

from gpu_helpers import MAX_ABS, Pair, compare, oracle_config

pytestmark = pytest.mark.gpu

SEED = 0x5EED_0123_4567_89AB


def check_sampled(gpu_logits, gpu_tok, orc_logits, T, pos, slot, where):
    z = sampling.sample_scores(orc_logits, T, pos, slot, SEED)
    top2 = np.sort(z)[-2:]
    margin = 2 * MAX_ABS / T + 1e-3
    if top2[1] - top2[0] > margin:
        assert gpu_tok == int(np.argmax(z)), f"{where}: sampled {gpu_tok} != oracle {int(np.argmax(z))}"
    # the GPU's token is the Gumbel-max of its own logits up to fp32 rounding
    zg = sampling.sample_scores(gpu_logits, T, pos, slot, SEED)
    assert zg[gpu_tok] >= zg.max() - 1e-3 * max(1.0, abs(zg.max())), where
    return int(np.argmax(z))


@pytest.mark.parametrize("T", [0.7, 1.5])
def test_tiny_sampled_decode_matches_oracle(cuda_dev, T):
    pair = Pair(TINY, 40)
    pair.mk.set_sampling(T, SEED)
    prompt = [int(t) for t in synth.prompt_tokens(TINY.vocab, 6)]
    tok, differs = prompt[0], 0
    for pos in range(20):
        gl, gt = pair.gpu_step(tok, pos)
        ol, ot_greedy = pair.orc.decode_step(tok, pos)
        compare(gl, int(np.argmax(gl)), ol, ot_greedy, f"T {T} pos {pos}")  # logits parity as usual
        ot = check_sampled(gl, gt, ol, T, pos, 0, f"T {T} pos {pos}")
        differs += ot != ot_greedy
        tok = prompt[pos + 1] if pos + 1 < len(prompt) else ot
    assert differs > 0  # the draws are not the greedy tokens
    # back to greedy
    pair.mk.set_sampling(0.0)
    gl, gt = pair.gpu_step(tok, 20)
    assert gt == int(np.argmax(gl))
    pair.close()


@pytest.mark.parametrize("pos,slot,seed", [(0, 0, 0), (129, 3, SEED), (8191, 7, (1 << 64) - 1)])
def test_kernel_philox_words_and_noise_match_the_oracle(cuda_dev, pos, slot, seed):
    # the epilogue's random stream, bit for bit, and its noise to fp32 rounding
    build()
    n = 4096
    words = torch.empty(n, dtype=torch.int32, device=cuda_dev)
    noise = torch.empty(n, dtype=torch.float32, device=cuda_dev)
    _lib.sampling_noise(n, pos, slot, seed, out_words=words, out_noise=noise)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(words.cpu().numpy().view(np.uint32), sampling.words(n, pos, slot, seed))
    np.testing.assert_allclose(noise.double().cpu().numpy(), sampling.gumbel(n, pos, slot, seed),
                               rtol=1e-5, atol=1e-5)


def test_kernel_noise_is_finite_at_the_boundary_words(cuda_dev):
    build()
    w = np.array([0x00000000, 0x000001FF, 0xFFFFFE00, 0xFFFFFFFF], dtype=np.uint32)
    words = torch.from_numpy(w.view(np.int32).copy()).to(cuda_dev)
    noise = torch.empty(4, dtype=torch.float32, device=cuda_dev)
    _lib.sampling_noise(4, 0, 0, 0, out_noise=noise, words=words)
    torch.cuda.synchronize()
    g = noise.double().cpu().numpy()
    assert np.isfinite(g).all(), g
    np.testing.assert_allclose(g, sampling.gumbel_from_word(w), rtol=1e-5, atol=1e-5)


def test_sampling_rejects_non_finite_temperature(cuda_dev):
    pair = Pair(TINY, 8)
    with pytest.raises(_lib.MKError):
        pair.mk.set_sampling(float("nan"))
    with pytest.raises(_lib.MKError):
        pair.mk.set_sampling(float("inf"))
    pair.close()


def test_llama1b_sampled_steps(cuda_dev):
    pair = Pair(LLAMA_1B, 8)
    pair.mk.set_sampling(0.8, SEED)
    prompt = [int(t) for t in synth.prompt_tokens(LLAMA_1B.vocab, 3)]
    tok = prompt[0]
    for pos in range(4):
        gl, gt = pair.gpu_step(tok, pos)
        ol, _ = pair.orc.decode_step(tok, pos)
        ot = check_sampled(gl, gt, ol, 0.8, pos, 0, f"pos {pos}")
        tok = prompt[pos + 1] if pos + 1 < len(prompt) else ot
    pair.close()


def test_tiny_batched_sampling_uses_each_sequence_slot(cuda_dev):
    # the fused batched step draws sequence b's noise on slot b
    build()
    dev = torch.device("cuda:0")
    B, T = 3, 0.9
    w = synth.make_weights(TINY, dev, 0)
    k, v = synth.kv_cache(TINY, 16, B, dev)
    mk = _lib.Megakernel(TINY, w, k, v)
    mk.set_sampling(T, SEED)
    hw = synth.host_weights(w)
    orcs = [oracle.OracleModel(oracle_config(TINY), hw, 16) for _ in range(B)]
    toks = torch.tensor([5, 5, 5], dtype=torch.int32, device=dev)  # same token: only the slot differs
    pos = torch.zeros(B, dtype=torch.int32, device=dev)
    out = torch.zeros(B, dtype=torch.int32, device=dev)
    logits = torch.empty(B, TINY.vocab, dtype=torch.float32, device=dev)
    cur = [5, 5, 5]
    for step in range(6):
        toks.copy_(torch.tensor(cur, dtype=torch.int32))
        pos.fill_(step)
        mk.step_batch(toks, pos, out, logits)
        torch.cuda.synchronize()
        assert mk.status() == 0
        gl = logits.double().cpu().numpy()
        gt = out.cpu().numpy().tolist()
        for b in range(B):
            ol, _ = orcs[b].decode_step(cur[b], step)
            cur[b] = check_sampled(gl[b], gt[b], ol, T, step, b, f"seq {b} step {step}")
    mk.close()


def check_filtered(gpu_logits, gpu_tok, T, top_k, top_p, pos, slot, where):
    """The GPU's filtered draw against the oracle's on the GPU's own logits.
    The kept set is computed in fp64 here and in fp32 on the GPU, so a
    nucleus whose cut falls within 1e-4 of top_p may differ by its last
    member; the draw must then come from the larger set. Elsewhere the token
    must be the oracle's, unless the two best noisy scores are within fp32
    rounding of each other."""
    hi = sampling.kept_set(gpu_logits, T, top_k, min(1.0, top_p + 1e-4))
    lo = sampling.kept_set(gpu_logits, T, top_k, max(1e-6, top_p - 1e-4))
    assert gpu_tok in set(hi.tolist()), f"{where}: token {gpu_tok} outside the kept set"
    if len(hi) == len(lo):
        want = sampling.sample_token_filtered(gpu_logits, T, pos, slot, SEED, top_k, top_p)
        s = gpu_logits[hi] / T + sampling.gumbel(gpu_logits.shape[0], pos, slot, SEED)[hi]
        top2 = np.sort(s)[-2:] if len(s) > 1 else np.array([-np.inf, s[0]])
        if top2[1] - top2[0] > 1e-4 * max(1.0, abs(top2[1])):
            assert gpu_tok == want, f"{where}: filtered draw {gpu_tok} != oracle {want}"
    return len(hi)


@pytest.mark.parametrize("top_k,top_p", [(1, 1.0), (5, 1.0), (64, 1.0), (0, 0.5), (40, 0.9), (0, 0.05)])
def test_tiny_filtered_draws_match_the_oracle(cuda_dev, top_k, top_p):
    T = 0.9
    pair = Pair(TINY, 40)
    pair.mk.set_sampling(T, SEED)
    pair.mk.set_sampling_filter(top_k, top_p)
    prompt = [int(t) for t in synth.prompt_tokens(TINY.vocab, 4)]
    tok, sizes = prompt[0], []
    for pos in range(16):
        gl, gt = pair.gpu_step(tok, pos)
        ol, ot_greedy = pair.orc.decode_step(tok, pos)
        compare(gl, int(np.argmax(gl)), ol, ot_greedy, f"pos {pos}")  # logits parity as usual
        sizes.append(check_filtered(gl, gt, T, top_k, top_p, pos, 0, f"k {top_k} p {top_p} pos {pos}"))
        if top_k == 1:
            assert gt == int(np.argmax(gl))
        tok = prompt[pos + 1] if pos + 1 < len(prompt) else gt
    if top_k > 0 and top_p >= 1.0:
        assert set(sizes) == {top_k}
    pair.mk.set_sampling_filter(0, 1.0)  # filter off again: the plain draw
    gl, gt = pair.gpu_step(tok, 16)
    check_sampled(gl, gt, pair.orc.decode_step(tok, 16)[0], T, 16, 0, "unfiltered")
    pair.close()


def test_llama1b_filtered_draws_match_the_oracle(cuda_dev):
    # 152 LM-head blocks of 844 rows each: the candidate merge at full size
    T = 0.7
    pair = Pair(LLAMA_1B, 8)
    pair.mk.set_sampling(T, SEED)
    prompt = [int(t) for t in synth.prompt_tokens(LLAMA_1B.vocab, 3)]
    tok = prompt[0]
    for pos, (k, p) in enumerate([(50, 0.9), (0, 0.3), (8, 1.0), (64, 0.99)]):
        pair.mk.set_sampling_filter(k, p)
        gl, gt = pair.gpu_step(tok, pos)
        check_filtered(gl, gt, T, k, p, pos, 0, f"k {k} p {p} pos {pos}")
        tok = prompt[pos + 1] if pos + 1 < len(prompt) else gt
    pair.close()


def test_fused_batch_filtered_draws_match_the_oracle(cuda_dev):
    # all sequences in one batched launch, then the draw kernels per sequence
    build()
    dev = torch.device("cuda:0")
    B, T = 3, 0.8
    w = synth.make_weights(TINY, dev, 0)
    k, v = synth.kv_cache(TINY, 16, B, dev)
    mk = _lib.Megakernel(TINY, w, k, v)
    mk.set_sampling(T, SEED)
    mk.set_sampling_filter(10, 0.8)
    toks = torch.tensor([5, 6, 7], dtype=torch.int32, device=dev)
    pos = torch.zeros(B, dtype=torch.int32, device=dev)
    out = torch.zeros(B, dtype=torch.int32, device=dev)
    logits = torch.empty(B, TINY.vocab, dtype=torch.float32, device=dev)
    for step in range(4):
        pos.fill_(step)
        mk.step_batch(toks, pos, out, logits)
        torch.cuda.synchronize()
        assert mk.status() == 0
        gl = logits.double().cpu().numpy()
        gt = out.cpu().numpy().tolist()
        for b in range(B):
            check_filtered(gl[b], gt[b], T, 10, 0.8, step, b, f"seq {b} step {step}")
        toks.copy_(out)
    mk.close()


def test_llama1b_fused_batch_filtered_draws(cuda_dev):
    # 8 sequences at the Llama-1B shape: 126 candidate lists of 1,024 entries
    # per sequence, drawn on each sequence's own slot and position
    build()
    dev = torch.device("cuda:0")
    B, T = 8, 0.7
    w = synth.make_weights(LLAMA_1B, dev, 0)
    k, v = synth.kv_cache(LLAMA_1B, 8, B, dev)
    mk = _lib.Megakernel(LLAMA_1B, w, k, v)
    mk.set_sampling(T, SEED)
    toks = torch.arange(100, 100 + B, dtype=torch.int32, device=dev)
    pos = torch.arange(B, dtype=torch.int32, device=dev) % 3
    out = torch.zeros(B, dtype=torch.int32, device=dev)
    logits = torch.empty(B, LLAMA_1B.vocab, dtype=torch.float32, device=dev)
    # top-k 1: 126 lists of one key, fewer keys than a run of 64
    for kk, pp in [(50, 0.9), (0, 0.5), (8, 1.0), (1, 1.0)]:
        mk.set_sampling_filter(kk, pp)
        mk.step_batch(toks, pos, out, logits)
        torch.cuda.synchronize()
        assert mk.status() == 0
        gl = logits.double().cpu().numpy()
        gt = out.cpu().numpy().tolist()
        for b in range(B):
            check_filtered(gl[b], gt[b], T, kk, pp, int(pos[b]), b, f"seq {b} k {kk} p {pp}")
        toks.copy_(out)
        pos += 1
    mk.close()


@pytest.mark.parametrize("top_k,top_p", [(0, 1.0), (40, 0.9)])
def test_prefill_token_is_drawn_like_the_decode_step(cuda_dev, top_k, top_p):
    # with sampling on, the prefill's token is the draw of its last position
    # (plain, then filtered) on that position's noise
    T, n = 0.8, 8
    pair = Pair(TINY, 16)
    pair.mk.set_sampling(T, SEED)
    pair.mk.set_sampling_filter(top_k, top_p)
    dev = torch.device("cuda:0")
    prompt = synth.prompt_tokens(TINY.vocab, n)
    out = torch.zeros(1, dtype=torch.int32, device=dev)
    logits = torch.empty(TINY.vocab, dtype=torch.float32, device=dev)
    pair.mk.prefill(prompt.to(dev), 0, out, logits)
    torch.cuda.synchronize()
    assert pair.mk.status() == 0
    for i in range(n):
        ol, _ = pair.orc.decode_step(int(prompt[i]), i)
    gl, gt = logits.double().cpu().numpy(), int(out.item())
    if top_k == 0 and top_p >= 1.0:
        check_sampled(gl, gt, ol, T, n - 1, 0, "prefill, plain draw")
    else:
        check_filtered(gl, gt, T, top_k, top_p, n - 1, 0, "prefill, filtered draw")
    # and without logits requested (an internal buffer takes them)
    out2 = torch.zeros(1, dtype=torch.int32, device=dev)
    pair.mk.prefill(prompt.to(dev), 0, out2)
    torch.cuda.synchronize()
    assert int(out2.item()) == gt
    pair.close()


@pytest.mark.parametrize("V", [1000, 4096, 50257, 128256])
@pytest.mark.parametrize("top_k,top_p", [(0, 1.0), (1, 1.0), (5, 1.0), (64, 1.0), (0, 0.9), (40, 0.2), (7, 0.95)])
def test_draw_from_logits_matches_the_oracle(cuda_dev, V, top_k, top_p):
    # the draw kernels on their own, over vocabularies that leave short runs
    # and short lists (1,000 entries: one slice of 1,024; 50,257: a ragged last
    # slice), with seeded N(0, 9) logits; two sequences on slots 0 and 1
    T, B = 0.9, 2
    rng = np.random.default_rng(V * 131 + top_k * 7 + int(top_p * 100))
    logits = (rng.standard_normal((B, V)) * 3.0).astype(np.float32)
    pos = np.array([7, 11], dtype=np.int32)
    out = torch.zeros(B, dtype=torch.int32, device=cuda_dev)
    _lib.draw_from_logits(torch.from_numpy(logits).to(cuda_dev), T, top_k, top_p,
                          torch.from_numpy(pos).to(cuda_dev), SEED, out)
    torch.cuda.synchronize()
    toks = out.cpu().numpy().tolist()
    for b in range(B):
        gl = logits[b].astype(np.float64)
        if top_k == 0 and top_p >= 1.0:  # the plain draw: the Gumbel-max of the logits
            z = sampling.sample_scores(gl, T, int(pos[b]), b, SEED)
            top2 = np.sort(z)[-2:]
            if top2[1] - top2[0] > 1e-4 * max(1.0, abs(top2[1])):
                assert toks[b] == int(np.argmax(z)), f"V {V} b {b}"
        else:
            check_filtered(gl, toks[b], T, top_k, top_p, int(pos[b]), b, f"V {V} k {top_k} p {top_p} b {b}")


def test_draw_from_logits_rejects_bad_arguments(cuda_dev):
    lg = torch.zeros(1, 10, device=cuda_dev)
    pos = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    for T, k, p in [(0.0, 0, 1.0), (float("nan"), 0, 1.0), (1.0, 65, 1.0), (1.0, 0, 0.0), (1.0, -1, 1.0)]:
        with pytest.raises(_lib.MKError) as e:
            _lib.draw_from_logits(lg, T, k, p, pos, SEED, out)
        assert e.value.code == _lib.MK_ERR_INVALID_ARG


def test_filter_arguments_are_checked(cuda_dev):
    pair = Pair(TINY, 8)
    for k, p in [(-1, 1.0), (65, 1.0), (5, 0.0), (5, 1.5), (5, float("nan"))]:
        with pytest.raises(_lib.MKError) as e:
            pair.mk.set_sampling_filter(k, p)
        assert e.value.code == _lib.MK_ERR_INVALID_ARG
    pair.close()


# 320,000 rows over 152 SMs at d_model 256: two LM-head instructions per SM
# (2,048 rows each at most), 304 blocks, more candidates than the last block
# sorts: the step picks greedily, writes its logits and the filter kernels
# draw after the launch.
WIDE = ModelShape("wide-vocab-320k", 2, 256, 4, 2, 64, 1024, 320000, 1e-5, 1e4)


@pytest.mark.parametrize("mode", ["mega", "unfused"])
def test_filtered_draw_after_the_launch_matches_the_oracle(cuda_dev, mode):
    instr, _, _ = _lib.plan_inspect(WIDE, torch.cuda.get_device_properties(0).multi_processor_count, 16)
    assert int((instr[:, 0] == 6).sum()) * 64 > 16384
    T = 0.8
    pair = Pair(WIDE, 16)
    pair.mk.set_sampling(T, SEED)
    prompt = [int(t) for t in synth.prompt_tokens(WIDE.vocab, 3)]
    tok = prompt[0]
    for pos, (k, p) in enumerate([(50, 0.9), (0, 0.3), (1, 1.0), (64, 0.99), (5, 1.0)]):
        pair.mk.set_sampling_filter(k, p)
        gl, gt = pair.gpu_step(tok, pos, mode)
        ol, ot = pair.orc.decode_step(tok, pos)
        compare(gl, int(np.argmax(gl)), ol, ot, f"pos {pos}")
        check_filtered(gl, gt, T, k, p, pos, 0, f"{mode} k {k} p {p} pos {pos}")
        if k == 1:
            assert gt == int(np.argmax(gl))
        tok = prompt[pos + 1] if pos + 1 < len(prompt) else gt
    # no logits asked for: the step keeps them in its own buffer
    pair.mk.set_sampling_filter(40, 0.9)
    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    pair.mk.step(tok, 5, out)
    gl, _ = pair.gpu_step(tok, 5, mode)  # the same position again: the same logits and noise
    torch.cuda.synchronize()
    assert pair.mk.status() == 0
    check_filtered(gl, int(out.item()), T, 40, 0.9, 5, 0, "no logits")
    pair.close()
