"""GPU parity of the activation-sparse FFN unit (mk_twell_down, mk_twell_ffn)
against the oracle's dense definitions (oracle.down_projection,
oracle.relu_glu) on the same seeded inputs.

Tolerance: every output is a sum of fp32 products of a bf16 weight and an
fp32 activation. The kernel adds them in a fixed tree: the rows one warp
visits (at most 32), then 8 warps, then the row blocks in 32 slices (at most
a few dozen blocks each here) and the 32 slice sums: fewer than 200
roundings of relative size 2^-24 on the way, so |y - y_oracle| <= 200 *
2^-24 * sum|terms| per element (the oracle itself is exact to far below
that). The gate/up dot
products of the FFN have d terms, lane by lane then over the warp: the same
bound with d / 64 + 5 + 1 roundings."""
import numpy as np
import pytest
import torch

import oracle
from decode_megakernel_llama_gb300 import _lib, synth
from decode_megakernel_llama_gb300.build import build

pytestmark = pytest.mark.gpu
U = 2.0 ** -24


def dec(bits):
    """bf16 bit patterns -> float64 (for the error bounds only)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def weights(rows, cols, seed, dev):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(rows, cols, generator=g) * 0.02).to(torch.bfloat16).to(dev)


def run_down(w_down, h):
    y = torch.full((w_down.shape[0],), float("nan"), dtype=torch.float32, device=w_down.device)
    _lib.twell_down(w_down.t().contiguous(), h, y)
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("F,d", [(8192, 2048), (1000, 256), (777, 3072), (3000, 1024), (64, 4096), (500, 2304),
                                 (33, 520)])
@pytest.mark.parametrize("sparsity", [0.0, 0.5, 0.9, 0.99, 1.0])
def test_sparse_down_matches_the_dense_definition(cuda_dev, F, d, sparsity):
    build()
    dev = torch.device("cuda:0")
    wd = weights(d, F, F + d, dev)  # the model's layout [d][F]
    h = synth.sparse_activations(F, sparsity, seed=F).to(dev)
    y = run_down(wd, h).double().cpu().numpy()
    bits = synth.bf16_bits(wd)
    hd = h.double().cpu().numpy()
    want = oracle.down_projection(bits, hd)
    scale = np.abs(dec(bits)) @ np.abs(hd)
    assert np.all(np.abs(y - want) <= 200 * U * scale + 1e-30), float(np.max(np.abs(y - want) - 200 * U * scale))
    if sparsity == 1.0:
        assert not np.any(y)  # nothing listed, nothing read: exact zeros


def test_sparse_down_is_bitwise_repeatable(cuda_dev):
    build()
    dev = torch.device("cuda:0")
    wd = weights(2048, 8192, 3, dev)
    h = synth.sparse_activations(8192, 0.7, seed=4).to(dev)
    a = run_down(wd, h)
    b = run_down(wd, h)
    assert torch.equal(a, b)


def test_sparse_down_rejects_bad_arguments(cuda_dev):
    build()
    dev = torch.device("cuda:0")
    h = torch.zeros(100, device=dev)
    for d in (4104, 100):  # wider than 4096; rows not a multiple of 16 bytes
        with pytest.raises(_lib.MKError) as e:
            _lib.twell_down(torch.zeros(100, d, dtype=torch.bfloat16, device=dev), h, torch.zeros(d, device=dev))
        assert e.value.code == -3
    raw = torch.zeros(100 * 2048 + 8, dtype=torch.bfloat16, device=dev)
    with pytest.raises(_lib.MKError) as e:  # weights not 16-byte aligned
        _lib.twell_down(raw[1:1 + 100 * 2048].view(100, 2048), h, torch.zeros(2048, device=dev))
    assert e.value.code == -1


@pytest.mark.parametrize("F,d", [(8192, 2048), (1000, 512)])
def test_relu_ffn_matches_the_oracle(cuda_dev, F, d):
    build()
    dev = torch.device("cuda:0")
    wg, wu, wd = weights(F, d, 11, dev), weights(F, d, 12, dev), weights(d, F, 13, dev)
    g = torch.Generator(device="cpu").manual_seed(14)
    x = torch.randn(d, generator=g).to(dev)
    h = torch.full((F,), float("nan"), device=dev)
    y = torch.full((d,), float("nan"), device=dev)
    _lib.twell_ffn(wg, wu, wd.t().contiguous(), x, h, y)
    torch.cuda.synchronize()
    xd = x.double().cpu().numpy()
    gb, ub = synth.bf16_bits(wg), synth.bf16_bits(wu)
    gd, ud = dec(gb), dec(ub)
    g_exact, u_exact = gd @ xd, ud @ xd
    tol = (d / 64 + 6) * U
    eg, eu = tol * (np.abs(gd) @ np.abs(xd)), tol * (np.abs(ud) @ np.abs(xd))
    want_h = oracle.relu_glu(gb, ub, xd)
    hg = h.double().cpu().numpy()
    # where the gate is clearly on or off both sides agree on zero / non-zero
    clear = np.abs(g_exact) > eg
    assert np.array_equal(hg[clear] == 0, want_h[clear] == 0)
    # value bound of max(g, 0) * u under the two dot products' error bounds
    bound = eg * np.abs(u_exact) + (np.maximum(g_exact, 0) + eg) * eu
    assert np.all(np.abs(hg - want_h) <= bound + 1e-30)
    assert 0.3 < float((hg == 0).mean()) < 0.7  # ReLU of random pre-activations: about half off
    # the down projection of the GPU's own h, against the dense definition
    yd = y.double().cpu().numpy()
    db = synth.bf16_bits(wd)
    want = oracle.down_projection(db, hg)
    scale = np.abs(dec(db)) @ np.abs(hg)
    assert np.all(np.abs(yd - want) <= 200 * U * scale + 1e-30)
