"""GPU parity of the W2A8 GEMV (mk_w2a8_gemv) against the oracle's
orc_matvec_w2a8 on the same fp32 input: both sides quantise the same fp32
values in fp32, so the activation codes and the integer dot products are
identical and the outputs differ only by the final fp32 scaling."""
import numpy as np
import pytest
import torch

import oracle
from decode_megakernel_llama_gb300 import _lib
from decode_megakernel_llama_gb300.build import build

pytestmark = pytest.mark.gpu


def ternary(rows, cols, seed, p_zero=1 / 3):
    rng = np.random.default_rng(seed)
    q = rng.choice(np.array([-1, 0, 1], dtype=np.int8), size=(rows, cols),
                   p=[(1 - p_zero) / 2, p_zero, (1 - p_zero) / 2])
    return q.astype(np.int8)


def run_gpu(q, beta, x32):
    rows, cols = q.shape
    dev = torch.device("cuda:0")
    packed = torch.from_numpy(_lib.w2_pack(q).view(np.int32)).to(dev)
    x = torch.from_numpy(x32).to(dev)
    y = torch.full((rows,), float("nan"), dtype=torch.float32, device=dev)
    _lib.w2a8_gemv(packed, beta, rows, cols, x, y)
    torch.cuda.synchronize()
    return y.double().cpu().numpy()


@pytest.mark.parametrize("rows,cols", [(100, 2048), (2048, 2048), (8192, 2048), (2048, 8192), (513, 4096),
                                       (77, 6144), (3072, 2048)])
def test_w2a8_gemv_matches_the_oracle(cuda_dev, rows, cols):
    build()
    rng = np.random.default_rng(rows * 7 + cols)
    q = ternary(rows, cols, rows + cols)
    for trial in range(3):
        x32 = (rng.normal(size=cols) * rng.uniform(0.05, 20)).astype(np.float32)
        if trial == 2:
            x32[rng.integers(0, cols)] = 400.0  # one outlier sets the scale
        beta = float(rng.uniform(0.01, 0.05))
        y = run_gpu(q, beta, x32)
        want = oracle.matvec_w2a8(q, beta, x32.astype(np.float64))
        scale = beta * np.abs(x32).max()
        np.testing.assert_allclose(y, want, rtol=2e-6, atol=1e-6 * scale)


def test_w2a8_gemv_zero_input_and_sparse_weights(cuda_dev):
    build()
    q = ternary(300, 2048, 1, p_zero=0.9)
    y = run_gpu(q, 0.03, np.zeros(2048, dtype=np.float32))
    assert (y == 0).all()
    x32 = np.linspace(-1, 1, 2048).astype(np.float32)
    np.testing.assert_allclose(run_gpu(q, 0.03, x32), oracle.matvec_w2a8(q, 0.03, x32.astype(np.float64)),
                               rtol=2e-6, atol=1e-7)


def test_w2a8_gemv_rejects_bad_sizes(cuda_dev):
    build()
    dev = torch.device("cuda:0")
    p = torch.zeros(16, 128, dtype=torch.int32, device=dev)
    x = torch.zeros(2048, dtype=torch.float32, device=dev)
    y = torch.zeros(16, dtype=torch.float32, device=dev)
    for cols in (1024, 3072, 16384):
        with pytest.raises(_lib.MKError):
            _lib.w2a8_gemv(p, 0.02, 16, cols, x, y)
