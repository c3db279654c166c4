"""Pins of the oracle's W2A8 projections (oracle.h: orc_w2a8_quantize,
orc_matvec_w2a8, orc_decode_step_w2a8): a hand-worked quantisation, exact
results when the input lies on the 8-bit grid, the rounding error bound
otherwise, invariance under power-of-two input scaling, and the whole W2A8
decode step against the pinned bf16 step on the same (dequantised) model."""
import numpy as np
import pytest

import oracle
from decode_megakernel_llama_gb300 import synth
from decode_megakernel_llama_gb300.configs import TINY


def test_quantize_hand_example():
    # s = 127 / max|x| = 127; -0.5 * 127 = -63.5 rounds half to even (-64);
    # 0.25 * 127 = 31.75 rounds to 32
    q, s = oracle.w2a8_quantize([1.0, -0.5, 0.25, 0.0])
    assert s == 127.0
    assert q.tolist() == [127, -64, 32, 0]
    q, s = oracle.w2a8_quantize([0.0, 0.0])  # all zero: the 1e-5 floor keeps s finite
    assert q.tolist() == [0, 0] and s == np.float32(127.0) / np.float32(1e-5)


def test_quantize_maps_the_absolute_maximum_to_127():
    rng = np.random.default_rng(1)
    for _ in range(20):
        x = rng.normal(size=777) * rng.uniform(0.01, 100)
        q, s = oracle.w2a8_quantize(x)
        i = int(np.argmax(np.abs(x)))
        assert abs(int(q[i])) == 127 and np.abs(q.astype(int)).max() == 127
        # each code is x * s rounded: within half a step
        assert np.all(np.abs(q - np.float32(x) * np.float32(s)) <= 0.5 + 1e-4)


def ternary(rows, cols, seed):
    return (np.random.default_rng(seed).integers(0, 3, size=(rows, cols)) - 1).astype(np.int8)


def test_matvec_is_exact_on_the_grid():
    # x = c / 8 with integer codes c and max |c| = 127: s = 8 exactly, the
    # codes are c, and y = beta * Wq x is exact in float64
    rng = np.random.default_rng(2)
    W = ternary(96, 512, 3)
    c = rng.integers(-127, 128, size=512)
    c[17] = 127
    x = c / 8.0
    beta = 0.0234375
    y = oracle.matvec_w2a8(W, beta, x)
    np.testing.assert_array_equal(y, beta * (W.astype(np.float64) @ x))


def test_matvec_error_is_within_the_rounding_bound():
    rng = np.random.default_rng(4)
    W = ternary(200, 1024, 5)
    for _ in range(10):
        x = rng.normal(size=1024)
        beta = float(rng.uniform(0.01, 0.05))
        y = oracle.matvec_w2a8(W, beta, x)
        _, s = oracle.w2a8_quantize(x)
        exact = beta * (W.astype(np.float64) @ x)
        bound = beta * np.abs(W).sum(axis=1) * (0.5 / s) * (1 + 1e-6) + 1e-12
        assert np.all(np.abs(y - exact) <= bound)
        assert np.abs(y - exact).max() > 0  # off the grid the codes do round


def test_matvec_scales_with_power_of_two_inputs():
    rng = np.random.default_rng(6)
    W = ternary(64, 256, 7)
    x = rng.normal(size=256)
    y = oracle.matvec_w2a8(W, 0.02, x)
    for f in (0.25, 2.0, 1024.0):
        np.testing.assert_array_equal(oracle.matvec_w2a8(W, 0.02, f * x), f * y)


def test_decode_step_tracks_the_bf16_step_on_the_dequantised_model():
    # beta is a bf16 value, so beta * Wq is an exact bf16 model; the W2A8
    # step differs from the bf16 step on it only by the 8-bit activation
    # rounding: a structural mistake (a wrong matrix, a dropped residual or
    # scale) breaks the agreement, the rounding does not
    w = synth.make_ternary_weights(TINY, "cpu", 0)
    hw = synth.host_ternary_weights(w)
    deq = {"embed": hw["embed"], "final_norm": hw["final_norm"], "layers": []}
    for lw in hw["layers"]:
        d = {"attn_norm": lw["attn_norm"], "mlp_norm": lw["mlp_norm"]}
        for m, b in zip(synth.W2_MATS, synth.W2_BETAS):
            d[m] = oracle.f64_to_bf16(lw[b] * lw[m].astype(np.float64))
        deq["layers"].append(d)
    cfg = oracle.OracleConfig(TINY.n_layers, TINY.d_model, TINY.n_heads, TINY.n_kv_heads, TINY.head_dim,
                              TINY.ffn_dim, TINY.vocab, TINY.rms_eps, TINY.rope_theta)
    a = oracle.OracleModelW2A8(cfg, hw, 16)
    b = oracle.OracleModel(cfg, deq, 16)
    for pos, tok in enumerate([5, 900, 31, 4000, 7, 7]):
        la, _ = a.decode_step(tok, pos)
        lb, _ = b.decode_step(tok, pos)
        cos = float(la @ lb / (np.linalg.norm(la) * np.linalg.norm(lb)))
        assert cos > 0.999, (pos, cos)
        assert np.abs(la - lb).max() < 0.05 * np.abs(lb).max()
    # the caches hold nearly the same keys and values
    for ca, cb in ((a.k_cache, b.k_cache), (a.v_cache, b.v_cache)):
        fa = (ca.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        fb = (cb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        assert np.abs(fa - fb).max() < 0.05 * np.abs(fb).max()
