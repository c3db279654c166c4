"""mk_decode_step_noalloc, the decode step for callers that cannot allocate
device memory (its scratch lives in a static device array of the library),
must give what the handle-based mk_decode_step gives. Collected last on
purpose: it runs after every other test, and also passes alone."""
import numpy as np
import pytest
import torch

from decode_megakernel_llama_gb300 import _lib, synth
from decode_megakernel_llama_gb300.build import build
from decode_megakernel_llama_gb300.configs import LLAMA_1B, TINY

from gpu_helpers import MAX_ABS, MIN_COS

pytestmark = pytest.mark.gpu


def _close(a: torch.Tensor, b: torch.Tensor):
    x, y = a.double().cpu().numpy(), b.double().cpu().numpy()
    assert np.abs(x - y).max() <= MAX_ABS
    assert float(x @ y / (np.linalg.norm(x) * np.linalg.norm(y))) >= MIN_COS


@pytest.mark.parametrize("shape,max_seq", [(TINY, 40), (LLAMA_1B, 64)])
def test_noalloc_step_matches_handle_step_twice(cuda_dev, shape, max_seq):
    build()
    dev = torch.device("cuda:0")
    w = synth.make_weights(shape, dev, 0)
    k1, v1 = synth.kv_cache(shape, max_seq, 1, dev)   # handle path's cache
    k2, v2 = synth.kv_cache(shape, max_seq, 1, dev)   # allocation-free path's cache
    mk = _lib.Megakernel(shape, w, k1, v1)
    l1 = torch.empty(shape.vocab, device=dev)
    l2 = torch.empty(shape.vocab, device=dev)
    t1 = torch.zeros(1, dtype=torch.int32, device=dev)
    t2 = torch.zeros(1, dtype=torch.int32, device=dev)
    tok = int(synth.prompt_tokens(shape.vocab, 1)[0])
    free_delta = None
    for pos in range(2):   # two calls in a row reuse the resident plan
        mk.step(tok, pos, t1, l1)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        _lib.decode_step_noalloc(shape, w, k2, v2, tok, pos, t2, l2)
        torch.cuda.synchronize()
        if pos == 1:  # after the warm-up call (module load, plan upload) nothing is allocated
            free_delta = free0 - torch.cuda.mem_get_info()[0]
        assert mk.status() == 0
        _close(l1, l2)
        assert int(t1.item()) == int(t2.item())
        tok = int(t1.item())
    assert free_delta == 0, f"the allocation-free call changed free device memory by {free_delta} bytes"
    torch.testing.assert_close(k1, k2, rtol=0, atol=0)
    mk.close()


def test_noalloc_rejects_oversized_model(cuda_dev):
    build()
    big = LLAMA_1B
    dev = torch.device("cuda:0")
    w = synth.make_weights(big, dev, 0)
    k, v = synth.kv_cache(big, 1, 1, dev)
    out = torch.zeros(1, dtype=torch.int32, device=dev)
    # a cache of 65536 positions needs a RoPE table beyond the 16 MiB array
    kbig = torch.empty((big.n_layers, 1, big.n_kv_heads, 65536, big.head_dim),
                       dtype=torch.bfloat16, device=dev)
    with pytest.raises(_lib.MKError) as e:
        _lib.decode_step_noalloc(big, w, kbig, kbig, 0, 0, out)
    assert e.value.code == _lib.MK_ERR_INVALID_ARG
    assert "scratch" in str(e.value)
