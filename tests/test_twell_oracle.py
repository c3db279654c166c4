"""Pins of the activation-sparse FFN oracle (oracle.relu_glu,
oracle.down_projection): a one-hot activation selects one column exactly,
numpy's float64 matrix product on the decoded weights, the exact zeros of the
ReLU gate, and invariance of the sum under a joint permutation of the hidden
units (the order in which a kernel visits the non-zero units changes no term)."""
import numpy as np

import oracle
from decode_megakernel_llama_gb300 import synth


def bf16_matrix(rows, cols, seed, scale=0.02):
    x = np.random.default_rng(seed).normal(size=(rows, cols)) * scale
    return oracle.f64_to_bf16(x) if rows * cols <= 4096 else _bf16_fast(x)


def _bf16_fast(x):
    # round to nearest even on the top 16 bits of the float32 encoding
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def test_one_hot_activation_selects_a_column():
    Wd = bf16_matrix(48, 64, 1)
    dec = oracle.bf16_to_f64(Wd)
    for i, v in ((0, 1.0), (17, -2.5), (63, 0.125)):
        h = np.zeros(64)
        h[i] = v
        np.testing.assert_array_equal(oracle.down_projection(Wd, h), dec[:, i] * v)


def test_down_projection_matches_numpy_on_sparse_activations():
    Wd = bf16_matrix(256, 1024, 2)
    dec = oracle.bf16_to_f64(Wd)
    for s in (0.0, 0.5, 0.9, 1.0):
        h = synth.sparse_activations(1024, s, seed=3).double().numpy()
        assert int((h == 0).sum()) == round(s * 1024)
        y = oracle.down_projection(Wd, h)
        np.testing.assert_allclose(y, dec @ h, rtol=1e-12, atol=1e-12)
        if s == 1.0:
            assert not y.any()


def test_relu_gate_zeros_exactly_where_the_gate_is_not_positive():
    Wg, Wu = bf16_matrix(512, 128, 4), bf16_matrix(512, 128, 5)
    x = np.random.default_rng(6).normal(size=128)
    h = oracle.relu_glu(Wg, Wu, x)
    g = oracle.bf16_to_f64(Wg) @ x
    u = oracle.bf16_to_f64(Wu) @ x
    np.testing.assert_array_equal(h == 0, (g <= 0) | (u == 0))
    np.testing.assert_allclose(h, np.maximum(g, 0) * u, rtol=1e-12, atol=1e-15)
    assert 0.3 < float((h == 0).mean()) < 0.7  # random weights: about half the units are off


def test_sum_is_invariant_under_a_joint_permutation_of_hidden_units():
    Wd = bf16_matrix(64, 512, 7)
    h = synth.sparse_activations(512, 0.75, seed=8).double().numpy()
    perm = np.random.default_rng(9).permutation(512)
    y = oracle.down_projection(Wd, h)
    yp = oracle.down_projection(np.ascontiguousarray(Wd[:, perm]), h[perm])
    np.testing.assert_allclose(yp, y, rtol=1e-12, atol=1e-14)
