"""Multi-token prefill (mk_prefill) and its tensor-core contraction
(mk_tc_gemm). The contraction is checked against a float64 product of the
same bf16 operands; the prefill against the oracle: the logits of the last
prompt position (both the oracle's incremental steps and its separately
coded full causal forward), the KV-cache rows of every prompt position, and
decoding that continues from the prefilled cache, teacher-forced."""
import numpy as np
import pytest
import torch

from decode_megakernel_llama_gb300 import _lib, synth
from decode_megakernel_llama_gb300.build import build
from decode_megakernel_llama_gb300.configs import LLAMA_1B, LLAMA_3B, TINY, WORKLOADS, ModelShape

from gpu_helpers import MAX_ABS, Pair, compare, teacher_forced

pytestmark = pytest.mark.gpu


def split(x: torch.Tensor):
    hi = x.to(torch.bfloat16)
    lo = (x - hi.float()).to(torch.bfloat16)
    return hi, lo


@pytest.mark.parametrize("M,K,N", [(128, 64, 32), (256, 256, 64), (96, 512, 5), (1000, 2048, 77),
                                   (3072, 2048, 128), (2048, 8192, 128), (8192, 2048, 200)])
def test_tc_gemm_matches_a_float64_product(cuda_dev, M, K, N):
    build()
    g = torch.Generator(device="cpu").manual_seed(M * 7 + K * 3 + N)
    w = (torch.randn(M, K, generator=g) * 0.02).to(torch.bfloat16)
    x = torch.randn(N, K, generator=g)
    hi, lo = split(x)
    exact = (hi.double() + lo.double()) @ w.double().T  # [N][M]
    scale = float((hi.double().abs() @ w.double().abs().T).max())
    wd, hd, ld = w.to(cuda_dev), hi.to(cuda_dev), lo.to(cuda_dev)
    y = torch.full((N, M), float("nan"), device=cuda_dev)
    _lib.tc_gemm(wd, hd, ld, y)
    err = (y.double().cpu() - exact).abs().max().item()
    assert err <= 2e-6 * scale, (err, scale)
    # with a residual added in place
    r = torch.randn(N, M, generator=g)
    y2 = r.to(cuda_dev)
    _lib.tc_gemm(wd, hd, ld, y2, r=y2)
    err2 = (y2.double().cpu() - (exact + r.double())).abs().max().item()
    assert err2 <= 2e-6 * scale + 1e-6, err2


def prefill_case(shape, n, max_seq, extra_decode, start_split=None):
    pair = Pair(shape, max_seq)
    dev = torch.device("cuda:0")
    prompt = synth.prompt_tokens(shape.vocab, n)
    out = torch.zeros(1, dtype=torch.int32, device=dev)
    logits = torch.empty(shape.vocab, dtype=torch.float32, device=dev)
    if start_split is None:
        pair.mk.prefill(prompt.to(dev), 0, out, logits)
    else:  # two prefills back to back: positions 0 .. s-1, then s .. n-1
        pair.mk.prefill(prompt[:start_split].to(dev), 0, out, logits)
        pair.mk.prefill(prompt[start_split:].to(dev), start_split, out, logits)
    torch.cuda.synchronize()
    assert pair.mk.status() == 0, _lib.load().mk_last_error()
    for i in range(n):
        ol, ot = pair.orc.decode_step(int(prompt[i]), i)
    gl = logits.double().cpu().numpy()
    compare(gl, int(out.item()), ol, ot, "prefill, last prompt position")
    # the cache rows of every prompt position, to rounding
    for gpu, orc in ((pair.k, pair.orc.k_cache), (pair.v, pair.orc.v_cache)):
        g = gpu[:, 0, :, :n].float().cpu().numpy()
        o = (orc[:, :, :n].astype(np.uint32) << 16).view(np.float32)
        assert np.abs(g - o).max() <= 2e-2 * max(1.0, np.abs(o).max()), np.abs(g - o).max()
    # decoding continues from the prefilled cache
    if extra_decode:
        teacher_forced(pair, [ot], extra_decode, start_pos=n)
    return pair, prompt, gl


def test_tiny_prefill_matches_the_oracle_and_decoding_continues(cuda_dev):
    wl = WORKLOADS["tiny"]
    pair, prompt, gl = prefill_case(TINY, wl.prompt_len, wl.max_seq, 8)
    # the oracle's separately coded full causal forward gives the same logits
    fl, _ = pair.orc.full_forward([int(t) for t in prompt])
    assert np.abs(gl - fl).max() <= MAX_ABS
    pair.close()


def test_tiny_prefill_in_two_parts_and_a_ragged_token_tile(cuda_dev):
    pair, _, _ = prefill_case(TINY, 37, 48, 3, start_split=13)
    pair.close()


def test_tiny_prefill_of_a_long_second_part(cuda_dev):
    # the second part starts at position 200 and attends to up to 300
    # positions: the cached rows of the first part and its own
    pair, _, _ = prefill_case(TINY, 300, 304, 2, start_split=200)
    pair.close()


def test_prefill_head_dim_128_over_several_key_tiles(cuda_dev):
    # head dim 128, three query heads per kv head (as the 3B shape), and a
    # second part that attends to up to 600 positions: three staged key tiles
    shape = ModelShape("hd128-g3", 2, 768, 6, 2, 128, 1536, 2048, 1e-5, 5e5)
    pair, _, _ = prefill_case(shape, 600, 608, 2, start_split=257)
    pair.close()


@pytest.mark.parametrize("n", [1, 33])
def test_tiny_prefill_of_one_token_and_of_one_past_the_short_prompt_path(cuda_dev, n):
    # 1 token: one token tile, one key; 33: the first length past the
    # short-prompt shapes (at most 32 tokens, every reduction split)
    pair, _, _ = prefill_case(TINY, n, 40, 2)
    pair.close()


def test_prefill_head_dim_128_short_prompt(cuda_dev):
    # head dim 128 through the short-prompt shapes (reductions split, q/k/v
    # partial sums added in the RoPE pass)
    shape = ModelShape("hd128-g3", 2, 768, 6, 2, 128, 1536, 2048, 1e-5, 5e5)
    pair, _, _ = prefill_case(shape, 20, 24, 2)
    pair.close()


def test_llama1b_prefill_of_the_workload_prompt(cuda_dev):
    wl = WORKLOADS["llama1b"]
    pair, _, _ = prefill_case(LLAMA_1B, wl.prompt_len, wl.max_seq, 4)
    pair.close()


def test_llama1b_prefill_of_a_short_prompt(cuda_dev):
    # at most 32 tokens: one token tile, every projection's reduction split
    # over up to 9 CTAs and summed in the RoPE and norm passes
    pair, _, _ = prefill_case(LLAMA_1B, 11, 24, 2)
    pair.close()


def test_llama3b_prefill_head_dim_128(cuda_dev):
    pair, _, _ = prefill_case(LLAMA_3B, 64, 72, 2)
    pair.close()


def test_prefill_rejects_bad_arguments_and_reports_bad_tokens(cuda_dev):
    pair = Pair(TINY, 16)
    dev = torch.device("cuda:0")
    out = torch.zeros(1, dtype=torch.int32, device=dev)
    with pytest.raises(_lib.MKError):
        pair.mk.prefill(torch.zeros(17, dtype=torch.int32, device=dev), 0, out)  # past max_seq
    with pytest.raises(_lib.MKError):
        pair.mk.prefill(torch.zeros(4, dtype=torch.int32, device=dev), 14, out)
    bad = torch.tensor([1, TINY.vocab + 3, 2], dtype=torch.int32, device=dev)
    pair.mk.prefill(bad, 0, out)
    torch.cuda.synchronize()
    assert pair.mk.status() == _lib.MK_ERR_INVALID_ARG
    # the handle works afterwards
    pair.mk.prefill(torch.tensor([1, 2, 3], dtype=torch.int32, device=dev), 0, out)
    torch.cuda.synchronize()
    assert pair.mk.status() == 0
    pair.close()
