"""Pins of the oracle's sampling step (oracle/sampling.py): Philox4x32-10
against the known-answer vectors published with the Random123 library
(tests/golden/philox4x32_10_kat.txt), and by properties (a bijection of the
counter for a fixed key, avalanche in key and counter, uniform output); the
word-to-uniform map stays strictly inside (0, 1) at both boundary words; the
Gumbel-max draw follows softmax(logits / T) and tends to the greedy token as
T -> 0."""
import os

import numpy as np
import pytest

from oracle import sampling

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def kat_vectors():
    rows = []
    for line in open(GOLDEN):
        line = line.split("#")[0].split()
        if line:
            rows.append([int(x, 16) for x in line])
    return rows


def test_philox_matches_the_published_known_answer_vectors():
    rows = kat_vectors()
    assert len(rows) == 3
    for r in rows:
        ctr, key, want = r[:4], r[4:6], r[6:10]
        got = sampling.philox4x32_10(*[np.array([c], dtype=np.uint64) for c in ctr], key[0], key[1])
        assert [int(g[0]) for g in got] == want, [hex(int(g[0])) for g in got]


def test_word_to_uniform_stays_inside_the_open_interval_at_the_boundaries():
    # the all-ones word was the failure case of a 24-bit mantissa recipe
    # ((2^24 - 1) + 1/2 rounds to 2^24 in fp32): 23 bits keep every step exact
    u = sampling.uniform_from_word(np.array([0x00000000, 0x000001FF, 0xFFFFFE00, 0xFFFFFFFF], dtype=np.uint32))
    assert u[0] == 2.0 ** -24 and u[1] == 2.0 ** -24
    assert u[2] == 1.0 - 2.0 ** -24 and u[3] == 1.0 - 2.0 ** -24
    # the same values in fp32 arithmetic are exact, so a float kernel gets them too
    top = np.float32(0xFFFFFFFF >> 9) + np.float32(0.5)
    assert float(top * np.float32(1.0 / 8388608.0)) == 1.0 - 2.0 ** -24
    g = sampling.gumbel_from_word(np.array([0, 0xFFFFFFFF], dtype=np.uint32))
    assert np.isfinite(g).all()
    assert g[0] < -2.8 and g[1] > 16.0  # -log(-log(2^-24)) and -log(2^-24 + ...)


def test_philox_is_a_bijection_of_the_counter():
    n = 1 << 16
    c0 = np.arange(n)
    out = sampling.philox4x32_10(c0, np.full(n, 7), np.full(n, 123456), np.full(n, 3), 0xDEADBEEF, 0x01234567)
    assert len(np.unique(np.stack(out, axis=1), axis=0)) == n


def _popcount(x: np.ndarray) -> np.ndarray:
    x = x.astype(np.uint64)
    c = np.zeros_like(x)
    for _ in range(32):
        c += x & np.uint64(1)
        x >>= np.uint64(1)
    return c


@pytest.mark.parametrize("which", ["key", "counter"])
def test_philox_flipping_one_input_bit_flips_half_the_output_bits(which):
    rng = np.random.default_rng(5)
    n = 4096
    c = [rng.integers(0, 1 << 32, n, dtype=np.uint64) for _ in range(4)]
    k0, k1 = 0x9A3B5C7D, 0x11223344
    a = sampling.philox4x32_10(*c, k0, k1)
    if which == "key":
        b = sampling.philox4x32_10(*c, k0 ^ (1 << 13), k1)
    else:
        c2 = list(c)
        c2[1] = c2[1] ^ np.uint64(1 << 20)
        b = sampling.philox4x32_10(*c2, k0, k1)
    flips = sum(_popcount(x ^ y) for x, y in zip(a, b))
    assert abs(float(flips.mean()) - 64.0) < 1.0, flips.mean()


def test_uniforms_are_uniform_in_the_open_interval():
    u = sampling.uniforms(1 << 16, position=17, slot=2, seed=99)
    assert u.min() > 0.0 and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 0.005
    counts, _ = np.histogram(u, bins=64, range=(0.0, 1.0))
    expected = len(u) / 64
    chi2 = float(((counts - expected) ** 2 / expected).sum())
    assert chi2 < 120.0, chi2  # 63 degrees of freedom: p < 1e-5 above ~115


def test_noise_depends_on_position_slot_and_seed():
    base = sampling.gumbel(64, 5, 0, 1)
    assert not np.allclose(base, sampling.gumbel(64, 6, 0, 1))
    assert not np.allclose(base, sampling.gumbel(64, 5, 1, 1))
    assert not np.allclose(base, sampling.gumbel(64, 5, 0, 2))
    assert not np.allclose(base, sampling.gumbel(64, 5, 0, 1 + (1 << 32)))
    np.testing.assert_array_equal(base, sampling.gumbel(64, 5, 0, 1))


@pytest.mark.parametrize("temperature", [1.0, 0.5, 2.0])
def test_gumbel_max_draws_follow_the_softmax(temperature):
    logits = np.array([0.0, 1.0, 2.0, -1.0, 0.5])
    n = 20000
    counts = np.zeros(len(logits))
    for pos in range(n):  # independent noise per position
        counts[sampling.sample_token(logits, temperature, pos, 3, 2024)] += 1
    z = logits / temperature
    p = np.exp(z - z.max())
    p /= p.sum()
    expected = n * p
    chi2 = float(((counts - expected) ** 2 / expected).sum())
    assert chi2 < 25.0, (chi2, counts, expected)  # 4 degrees of freedom: p < 1e-4 above ~23.5


def test_small_temperature_is_greedy_and_nonpositive_is_greedy():
    rng = np.random.default_rng(11)
    for pos in range(50):
        logits = rng.normal(size=300)
        top = int(np.argmax(logits))
        assert sampling.sample_token(logits, 0.0, pos, 0, 7) == top
        assert sampling.sample_token(logits, -1.0, pos, 0, 7) == top
        gap = np.sort(logits)[-1] - np.sort(logits)[-2]
        if gap > 1e-3:
            assert sampling.sample_token(logits, 1e-5, pos, 0, 7) == top


def test_greedy_ties_go_to_the_lowest_index():
    assert sampling.sample_token(np.array([1.0, 3.0, 3.0, 1.0]), 0.0, 0, 0, 0) == 1


# ---- top-k / top-p (oracle/sampling.py: candidates, kept_set, sample_token_filtered)

def test_top_k_1_is_greedy_at_any_temperature():
    rng = np.random.default_rng(21)
    for pos in range(40):
        z = rng.normal(size=500)
        z[rng.integers(0, 500)] = z.max()  # a tie at the top: the lower index wins
        top = int(np.argmax(z))
        for T in (0.3, 1.0, 4.0):
            assert sampling.sample_token_filtered(z, T, pos, 1, 99, top_k=1) == top


def test_no_filter_and_a_full_top_k_equal_the_plain_draw():
    rng = np.random.default_rng(22)
    for pos in range(40):
        z = rng.normal(size=64) * 3
        plain = sampling.sample_token(z, 0.9, pos, 2, 5)
        assert sampling.sample_token_filtered(z, 0.9, pos, 2, 5) == plain
        assert sampling.sample_token_filtered(z, 0.9, pos, 2, 5, top_k=64) == plain
        assert sampling.sample_token_filtered(z, 0.9, pos, 2, 5, top_k=64, top_p=1.0) == plain


def test_candidates_break_ties_by_the_lower_index():
    z = np.array([1.0, 5.0, 3.0, 5.0, 3.0, 3.0, 0.0])
    assert sampling.candidates(z, 4).tolist() == [1, 3, 2, 4]
    assert sampling.kept_set(z, 1.0, 3, 1.0).tolist() == [1, 3, 2]


@pytest.mark.parametrize("p", [0.05, 0.3, 0.5, 0.9, 0.999])
def test_nucleus_is_the_smallest_set_reaching_the_mass(p):
    # brute force over every subset of a small vocabulary: the kept set has
    # the fewest members of any subset whose mass reaches p (a prefix of the
    # sorted order attains that minimum), and it is a prefix of the order
    import itertools
    rng = np.random.default_rng(int(p * 1000))
    for _ in range(20):
        z = rng.normal(size=8) * 2
        T = float(rng.uniform(0.5, 2.0))
        e = np.exp((z - z.max()) / T)
        prob = e / e.sum()
        keep = sampling.kept_set(z, T, 0, p)
        best = min(len(s) for r in range(1, 9) for s in itertools.combinations(range(8), r)
                   if prob[list(s)].sum() >= p - 1e-12)
        assert len(keep) == best
        assert prob[keep].sum() >= p - 1e-12
        assert prob[keep[:-1]].sum() < p  # minimal: without its last member it falls short
        assert keep.tolist() == sampling.candidates(z, len(keep)).tolist()


def test_top_p_acts_within_the_capped_candidates():
    # 1000 equal logits: the nucleus of mass 0.9 would need 900 tokens, the
    # cap keeps it to the MAX_TOP_K lowest indices
    z = np.zeros(1000)
    keep = sampling.kept_set(z, 1.0, 0, 0.9)
    assert keep.tolist() == list(range(int(np.ceil(0.9 * sampling.MAX_TOP_K))))


@pytest.mark.parametrize("top_k,top_p", [(3, 1.0), (0, 0.6), (4, 0.8)])
def test_filtered_draws_follow_the_renormalised_softmax(top_k, top_p):
    z = np.array([0.0, 1.0, 2.0, -1.0, 0.5, 1.5])
    T = 0.8
    keep = sampling.kept_set(z, T, top_k, top_p)
    n = 20000
    counts = np.zeros(len(z))
    for pos in range(n):
        counts[sampling.sample_token_filtered(z, T, pos, 0, 77, top_k, top_p)] += 1
    assert counts[np.setdiff1d(np.arange(len(z)), keep)].sum() == 0
    e = np.exp(z[keep] / T)
    expected = n * e / e.sum()
    chi2 = float(((counts[keep] - expected) ** 2 / expected).sum())
    assert chi2 < 25.0, (chi2, counts, expected)  # <= 5 degrees of freedom: p < 1e-4 above ~20.5
