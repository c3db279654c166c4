"""Pins of the fp64 CPU oracle against facts that do not come from the oracle.

Each test checks one oracle function against a closed form, an invariant, a
library routine (numpy / scipy / torch in float64) or a separately coded
computation, chosen so that a dropped term, a wrong sign or index, or a
transposed operand in the oracle fails at least one of them. CPU only.
"""
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from decode_megakernel_llama_gb300.configs import TINY, ModelShape
from decode_megakernel_llama_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_bf16(shape, std=1.0, seed=0):
    g = torch.Generator().manual_seed(seed)
    return synth.bf16_bits((torch.randn(shape, generator=g) * std).to(torch.bfloat16))


def bits_to_f64(bits):
    """Library widening: torch reinterprets the bits as bfloat16."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


# ---- bf16 format ------------------------------------------------------------

def test_bf16_golden_values():
    rows = []
    with open(os.path.join(GOLDEN, "bf16_values.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                val, bits = line.split()[:2]
                rows.append((float(val), int(bits, 16)))
    assert len(rows) >= 10
    for val, bits in rows:
        assert int(oracle.f64_to_bf16([val])[0]) == bits, (val, hex(bits))
        back = oracle.bf16_to_f64(np.array([bits], dtype=np.uint16))[0]
        # exact values round-trip; ties map to the even neighbour
        assert back == bits_to_f64(np.array([bits], dtype=np.uint16))[0]


def test_bf16_rounding_matches_torch_on_float32_values():
    # For inputs that are binary32 values, rounding from double equals the
    # library's float32 -> bfloat16 round-to-nearest-even.
    g = torch.Generator().manual_seed(5)
    x32 = torch.randn(4000, generator=g, dtype=torch.float32) * torch.exp(
        torch.randn(4000, generator=g) * 4)
    ref = synth.bf16_bits(x32.to(torch.bfloat16))
    got = oracle.f64_to_bf16(x32.double().numpy())
    np.testing.assert_array_equal(got, ref)


def test_bf16_widening_matches_library():
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    finite = ~np.isnan(bits_to_f64(bits))
    np.testing.assert_array_equal(oracle.bf16_to_f64(bits)[finite], bits_to_f64(bits)[finite])


# ---- RMSNorm ----------------------------------------------------------------

@pytest.mark.parametrize("c", [0.5, -3.0, 1e-3])
def test_rmsnorm_constant_vector_closed_form(c):
    n, eps = 64, 1e-5
    g = rand_bf16((n,), 0.3, seed=1)
    out = oracle.rmsnorm(np.full(n, c), g, eps)
    expect = bits_to_f64(g) * c / math.sqrt(c * c + eps)
    np.testing.assert_allclose(out, expect, rtol=1e-13, atol=0)


def test_rmsnorm_unit_gain_has_unit_rms_and_is_scale_invariant():
    x = np.random.default_rng(0).standard_normal(257) * 7.0
    ones = oracle.f64_to_bf16(np.ones(257))
    y = oracle.rmsnorm(x, ones, 0.0)
    assert abs(math.sqrt(np.mean(y * y)) - 1.0) < 1e-13
    np.testing.assert_allclose(oracle.rmsnorm(3.0 * x, ones, 0.0), y, rtol=1e-13)
    # eps sits inside the square root: mean-square 1 vector -> 1/sqrt(1+eps)
    z = np.ones(16)
    np.testing.assert_allclose(oracle.rmsnorm(z, ones[:16], 0.25), z / math.sqrt(1.25), rtol=1e-15)


# ---- matvec -------------------------------------------------------------------

@pytest.mark.parametrize("rows,cols", [(3, 5), (7, 1), (1, 9), (33, 64)])
def test_matvec_matches_numpy(rows, cols):
    W = rand_bf16((rows, cols), seed=rows * 100 + cols)
    x = np.random.default_rng(rows).standard_normal(cols)
    np.testing.assert_allclose(oracle.matvec(W, x), bits_to_f64(W) @ x, rtol=1e-12, atol=1e-12)


# ---- RoPE ---------------------------------------------------------------------

def test_rope_position_zero_is_identity():
    v = np.random.default_rng(1).standard_normal(64)
    np.testing.assert_array_equal(oracle.rope(v, 0, 1e4), v)


@pytest.mark.parametrize("hd,theta", [(64, 1e4), (128, 5e5), (8, 10.0)])
def test_rope_preserves_norm_and_pair_norms(hd, theta):
    v = np.random.default_rng(hd).standard_normal(hd)
    r = oracle.rope(v, 1234, theta)
    h = hd // 2
    np.testing.assert_allclose(np.hypot(r[:h], r[h:]), np.hypot(v[:h], v[h:]), rtol=1e-12)


@pytest.mark.parametrize("hd,theta", [(64, 1e4), (128, 5e5)])
def test_rope_rotation_angle_per_pair(hd, theta):
    # Pair (i, i+hd/2) is rotated counter-clockwise by pos * theta^(-2i/hd):
    # measure the angle with atan2 and compare with that frequency schedule.
    h = hd // 2
    e = np.zeros(hd)
    e[:h] = 1.0  # every pair starts on the positive real axis
    pos = 3
    r = oracle.rope(e, pos, theta)
    ang = np.arctan2(r[h:], r[:h])
    want = np.angle(np.exp(1j * pos * theta ** (-2.0 * np.arange(h) / hd)))
    np.testing.assert_allclose(ang, want, atol=1e-12)


def test_rope_relative_position_dot_product():
    rng = np.random.default_rng(7)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    base = oracle.rope(q, 17, 1e4) @ oracle.rope(k, 5, 1e4)
    for shift in (1, 100, 4000):
        d = oracle.rope(q, 17 + shift, 1e4) @ oracle.rope(k, 5 + shift, 1e4)
        assert abs(d - base) < 1e-9 * max(1.0, abs(base))


# ---- SiLU / softmax --------------------------------------------------------

def test_silu_special_values():
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(1.0) - scipy.special.expit(1.0)) < 1e-15
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12
    assert abs(oracle.silu(-40.0)) < 1e-15
    for z in (0.3, 2.5, -7.0):  # silu(z) - silu(-z) = z
        assert abs(oracle.silu(z) - oracle.silu(-z) - z) < 1e-14


def test_softmax_matches_scipy_and_sums_to_one():
    s = np.random.default_rng(3).standard_normal(50) * 10
    p = oracle.softmax(s)
    assert abs(p.sum() - 1.0) < 1e-12
    np.testing.assert_allclose(p, scipy.special.softmax(s), rtol=1e-12)
    np.testing.assert_allclose(oracle.softmax(s + 1000.0), p, rtol=1e-12)


# ---- attention ----------------------------------------------------------------

def test_attention_single_position_returns_v():
    K, V = rand_bf16((1, 64), seed=11), rand_bf16((1, 64), seed=12)
    q = np.random.default_rng(0).standard_normal(64) * 10
    np.testing.assert_array_equal(oracle.attend(q, K, V), bits_to_f64(V)[0])


def test_attention_equal_scores_give_mean_of_v():
    V = rand_bf16((9, 64), seed=13)
    K = np.tile(rand_bf16((1, 64), seed=14), (9, 1))
    q = np.random.default_rng(1).standard_normal(64)
    np.testing.assert_allclose(oracle.attend(q, K, V), bits_to_f64(V).mean(0), rtol=1e-12, atol=1e-14)


def test_attention_scale_is_inverse_sqrt_head_dim():
    # two keys: scores s0 = c*c/sqrt(hd) and s1 = 0 -> weights expit(s0)
    hd, c = 16, 3.0
    K = np.zeros((2, hd)); K[0, 0] = c
    V = np.zeros((2, hd)); V[0, 1] = 1.0; V[1, 2] = 1.0
    q = np.zeros(hd); q[0] = c
    o = oracle.attend(q, oracle.f64_to_bf16(K), oracle.f64_to_bf16(V))
    w0 = scipy.special.expit(c * c / math.sqrt(hd))
    np.testing.assert_allclose([o[1], o[2]], [w0, 1 - w0], rtol=1e-13)


def test_attention_matches_scipy_softmax_weighting():
    T, hd = 37, 64
    K, V = rand_bf16((T, hd), seed=21), rand_bf16((T, hd), seed=22)
    q = np.random.default_rng(2).standard_normal(hd) * 3
    p = scipy.special.softmax(bits_to_f64(K) @ q / math.sqrt(hd))
    np.testing.assert_allclose(oracle.attend(q, K, V), p @ bits_to_f64(V), rtol=1e-11, atol=1e-13)


def test_argmax_lowest_index_on_ties():
    assert oracle.argmax([1.0, 3.0, 3.0, 2.0]) == 1
    assert oracle.argmax([5.0, 5.0]) == 0
    assert oracle.argmax([-1.0, -0.5, -0.5]) == 1


# ---- MLP block ----------------------------------------------------------------

SMALL = ModelShape("small", 2, 32, 4, 2, 8, 48, 97, 1e-5, 1e4)


def small_model(shape=SMALL, seed=0, max_seq=16):
    w = synth.host_weights(synth.make_weights(shape, "cpu", seed))
    cfg = oracle.OracleConfig(shape.n_layers, shape.d_model, shape.n_heads, shape.n_kv_heads,
                              shape.head_dim, shape.ffn_dim, shape.vocab, shape.rms_eps,
                              shape.rope_theta)
    return cfg, w, oracle.OracleModel(cfg, w, max_seq)


def mlp_delta(lw, x, eps=1e-5):
    import ctypes
    L = oracle._Layer()
    keep = {k: np.ascontiguousarray(v) for k, v in lw.items()}
    for k, v in keep.items():
        setattr(L, k, oracle._p16(v))
    xx = np.ascontiguousarray(x, dtype=np.float64).copy()
    oracle.lib().orc_mlp_block.argtypes = [ctypes.POINTER(oracle._Layer), ctypes.c_int,
                                           ctypes.c_int, ctypes.c_double, oracle._PD]
    oracle.lib().orc_mlp_block(ctypes.byref(L), x.size, lw["w_gate"].shape[0], eps, oracle._pd(xx))
    return xx - x


def test_mlp_is_linear_in_up_and_zero_without_down():
    _, w, _ = small_model()
    lw = dict(w["layers"][0])
    x = np.random.default_rng(4).standard_normal(SMALL.d_model)
    d1 = mlp_delta(lw, x)
    up2 = oracle.f64_to_bf16(2.0 * bits_to_f64(lw["w_up"]))
    d2 = mlp_delta(dict(lw, w_up=up2), x)
    # silu(g) * (2u) = 2 silu(g) u; only the residual add (x + t) - x rounds
    np.testing.assert_allclose(d2, 2.0 * d1, rtol=0, atol=4 * np.finfo(float).eps * np.max(np.abs(x)))
    zero = np.zeros_like(lw["w_down"])
    assert np.all(mlp_delta(dict(lw, w_down=zero), x) == 0.0)


def test_mlp_gate_goes_through_silu_not_up():
    # A strongly negative gate closes the unit (silu -> 0); a strongly negative
    # up projection does not.
    _, w, _ = small_model()
    lw = dict(w["layers"][0])
    x = np.abs(np.random.default_rng(5).standard_normal(SMALL.d_model)) + 0.5
    ones_g = oracle.f64_to_bf16(np.ones(SMALL.d_model))
    lw["mlp_norm"] = ones_g
    big_neg = oracle.f64_to_bf16(np.full((SMALL.ffn_dim, SMALL.d_model), -8.0))
    closed = mlp_delta(dict(lw, w_gate=big_neg), x)
    assert np.max(np.abs(closed)) < 1e-10
    open_ = mlp_delta(dict(lw, w_up=big_neg), x)
    assert np.max(np.abs(open_)) > 1e-3


# ---- whole decode step ------------------------------------------------------------

def test_zero_blocks_reduce_to_embedding_lm_head():
    # With every projection zero the residual stream stays E[tok], so the
    # logits are E @ (RMSNorm(E[tok]) * g_final), computed here with numpy.
    cfg, w, _ = small_model()
    for lw in w["layers"]:
        for k in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down"):
            lw[k] = np.zeros_like(lw[k])
    m = oracle.OracleModel(cfg, w, 8)
    E = bits_to_f64(w["embed"])
    gf = bits_to_f64(w["final_norm"])
    for pos, tok in enumerate([3, 96, 0]):
        logits, t = m.decode_step(tok, pos)
        x = E[tok]
        xh = x / np.sqrt(np.mean(x * x) + cfg.rms_eps) * gf
        np.testing.assert_allclose(logits, E @ xh, rtol=1e-12, atol=1e-14)
        assert t == int(np.argmax(E @ xh))


def test_first_position_ignores_query_and_key_weights():
    # At position 0 the only attended position is the token itself, whose
    # softmax weight is 1 whatever q and k are.
    cfg, w, m1 = small_model()
    l1, _ = m1.decode_step(5, 0)
    w2 = {**w, "layers": [dict(lw, wq=rand_bf16(lw["wq"].shape, 0.5, 99),
                               wk=rand_bf16(lw["wk"].shape, 0.5, 98)) for lw in w["layers"]]}
    m2 = oracle.OracleModel(cfg, w2, 16)
    l2, _ = m2.decode_step(5, 0)
    np.testing.assert_array_equal(l1, l2)
    # ...but at position 1 they matter
    a, _ = m1.decode_step(7, 1)
    b, _ = m2.decode_step(7, 1)
    assert np.max(np.abs(a - b)) > 1e-6


def test_decode_ignores_cache_beyond_position():
    cfg, w, m1 = small_model()
    _, _, m2 = small_model()
    m2.k_cache[:] = rand_bf16(m2.k_cache.shape, 3.0, 7)
    m2.v_cache[:] = rand_bf16(m2.v_cache.shape, 3.0, 8)
    for pos, tok in enumerate([1, 2, 3, 4]):
        a, _ = m1.decode_step(tok, pos)
        b, _ = m2.decode_step(tok, pos)
        np.testing.assert_array_equal(a, b)


def test_incremental_decode_equals_full_causal_forward():
    cfg, w, m = small_model()
    toks = [11, 50, 3, 3, 96, 0, 42]
    for n in range(1, len(toks) + 1):
        inc, ti = m.decode_step(toks[n - 1], n - 1)
        full, tf = m.full_forward(toks[:n])
        np.testing.assert_allclose(inc, full, rtol=1e-12, atol=1e-12)
        assert ti == tf


def test_gqa_equals_mha_with_repeated_kv_heads():
    # Contiguous groups: query head h reads kv head h // G. Repeating each kv
    # head's rows G times (in place) gives an MHA model with identical output.
    cfg, w, m = small_model()
    G = SMALL.n_heads // SMALL.n_kv_heads
    hd = SMALL.head_dim
    rep = lambda W: np.repeat(W.reshape(SMALL.n_kv_heads, hd, -1), G, axis=0).reshape(-1, W.shape[1])
    w_mha = {**w, "layers": [dict(lw, wk=rep(lw["wk"]), wv=rep(lw["wv"])) for lw in w["layers"]]}
    mha = ModelShape("mha", SMALL.n_layers, SMALL.d_model, SMALL.n_heads, SMALL.n_heads,
                     hd, SMALL.ffn_dim, SMALL.vocab)
    cfg2 = oracle.OracleConfig(mha.n_layers, mha.d_model, mha.n_heads, mha.n_kv_heads,
                               mha.head_dim, mha.ffn_dim, mha.vocab, mha.rms_eps, mha.rope_theta)
    m2 = oracle.OracleModel(cfg2, w_mha, 16)
    for pos, tok in enumerate([9, 8, 7, 6]):
        a, _ = m.decode_step(tok, pos)
        b, _ = m2.decode_step(tok, pos)
        np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-13)
    # the other mapping (h % Hkv) would differ: swapping kv heads changes output
    w_sw = {**w, "layers": [dict(lw, wk=lw["wk"].reshape(SMALL.n_kv_heads, hd, -1)[::-1].reshape(-1, SMALL.d_model).copy(),
                                 wv=lw["wv"].reshape(SMALL.n_kv_heads, hd, -1)[::-1].reshape(-1, SMALL.d_model).copy())
                            for lw in w["layers"]]}
    m3 = oracle.OracleModel(cfg, w_sw, 16)
    m4 = oracle.OracleModel(cfg, w, 16)
    outs = []
    for mm in (m3, m4):
        mm.decode_step(9, 0)
        outs.append(mm.decode_step(8, 1)[0])
    assert np.max(np.abs(outs[0] - outs[1])) > 1e-6


def test_kv_cache_holds_bf16_post_rope_keys():
    # After a step at pos p, cache row p of layer 0 holds bf16(RoPE(Wk xh, p))
    # and bf16(Wv xh), built here from the oracle's pinned primitives.
    cfg, w, m = small_model()
    tok, pos = 17, 3
    m.decode_step(tok, pos)
    E = w["embed"]
    lw = w["layers"][0]
    x = bits_to_f64(E[tok])
    xh = oracle.rmsnorm(x, lw["attn_norm"], cfg.rms_eps)
    k = oracle.matvec(lw["wk"], xh).reshape(cfg.n_kv_heads, cfg.head_dim)
    v = oracle.matvec(lw["wv"], xh).reshape(cfg.n_kv_heads, cfg.head_dim)
    for h in range(cfg.n_kv_heads):
        np.testing.assert_array_equal(m.k_cache[0, h, pos], oracle.f64_to_bf16(oracle.rope(k[h], pos, cfg.rope_theta)))
        np.testing.assert_array_equal(m.v_cache[0, h, pos], oracle.f64_to_bf16(v[h]))


def test_decode_rejects_bad_arguments():
    _, _, m = small_model()
    with pytest.raises(ValueError):
        m.decode_step(SMALL.vocab, 0)
    with pytest.raises(ValueError):
        m.decode_step(0, 16)
    with pytest.raises(ValueError):
        m.decode_step(-1, 0)


def test_tiny_config_runs_and_is_deterministic():
    w = synth.host_weights(synth.make_weights(TINY, "cpu", 0))
    cfg = oracle.OracleConfig(TINY.n_layers, TINY.d_model, TINY.n_heads, TINY.n_kv_heads,
                              TINY.head_dim, TINY.ffn_dim, TINY.vocab, TINY.rms_eps, TINY.rope_theta)
    a = oracle.OracleModel(cfg, w, 8)
    b = oracle.OracleModel(cfg, w, 8)
    oracle.set_threads(1)
    la, ta = a.decode_step(1, 0)
    oracle.set_threads(4)
    lb, tb = b.decode_step(1, 0)
    oracle.set_threads(0)
    np.testing.assert_array_equal(la, lb)
    assert ta == tb and np.isfinite(la).all()
