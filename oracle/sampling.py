"""Sampling step of the oracle: a draw from softmax(logits / T) by the
Gumbel-max rule with counter-based noise.

TEST INFRASTRUCTURE ONLY, like the rest of this package: the test suite is
its only user. It shares no code with the CUDA library; the library's
sampling epilogue is a separate implementation of the same two published
definitions.

* Philox4x32-10 (J. Salmon, M. Moraes, R. Dror, D. Shaw, "Parallel random
  numbers: as easy as 1, 2, 3", SC'11, section 3): a 128-bit counter and a
  64-bit key; each of ten rounds multiplies counter words 0 and 2 by the
  constants M0 = 0xD2511F53 and M1 = 0xCD9E8D57 into 64-bit products and
  recombines the halves with words 1 and 3 and the key, which is then
  bumped by the Weyl constants W0 = 0x9E3779B9 and W1 = 0xBB67AE85.
* The Gumbel-max rule (E. J. Gumbel, 1954; used for sampling by Maddison,
  Tarlow, Minka, "A* sampling", NIPS 2014): with g_i = -log(-log(u_i)) for
  independent uniforms u_i, argmax_i(z_i + g_i) is distributed as
  softmax(z).

The noise of vocabulary entry i for the sequence on KV slot s at position
pos is u_i = (top 23 bits of output word 0 of Philox(counter (i, pos, s, 0),
key (seed mod 2^32, seed div 2^32)) + 1/2) / 2^23, which lies strictly
inside (0, 1) for every word (at most 1 - 2^-24), and the sampled token is
argmax_i(logit_i / T + g_i), lowest index on ties. Philox is pinned to the
known-answer vectors published with the Random123 library (the SC'11
authors' distribution) and by properties (bijectivity for a fixed key, key
sensitivity, uniformity); the sampler by a T -> 0 limit (greedy) and the
softmax law of the draws.
"""
from __future__ import annotations

import numpy as np

M0, M1 = 0xD2511F53, 0xCD9E8D57
W0, W1 = 0x9E3779B9, 0xBB67AE85
_MASK = 0xFFFFFFFF


def philox4x32_10(c0, c1, c2, c3, k0: int, k1: int) -> tuple:
    """All four output words of Philox4x32-10, elementwise over counter
    arrays (any integer arrays of one shape, values < 2^32)."""
    c = [np.asarray(x, dtype=np.uint64) & _MASK for x in (c0, c1, c2, c3)]
    k0, k1 = np.uint64(k0 & _MASK), np.uint64(k1 & _MASK)
    for _ in range(10):
        p0 = c[0] * np.uint64(M0)           # exact: both factors < 2^32
        p1 = c[2] * np.uint64(M1)
        hi0, lo0 = p0 >> np.uint64(32), p0 & np.uint64(_MASK)
        hi1, lo1 = p1 >> np.uint64(32), p1 & np.uint64(_MASK)
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
        k0 = (k0 + np.uint64(W0)) & np.uint64(_MASK)
        k1 = (k1 + np.uint64(W1)) & np.uint64(_MASK)
    return tuple(x.astype(np.uint32) for x in c)


def words(n: int, position: int, slot: int, seed: int) -> np.ndarray:
    """Output word 0 of Philox for counters (i, position, slot, 0), i = 0..n-1."""
    i = np.arange(n, dtype=np.uint64)
    return philox4x32_10(i, np.full(n, position), np.full(n, slot), np.zeros(n), seed & _MASK,
                         (seed >> 32) & _MASK)[0]


def uniform_from_word(w) -> np.ndarray:
    """(top 23 bits of w + 1/2) / 2^23 as float64: in [2^-24, 1 - 2^-24]."""
    w = np.asarray(w, dtype=np.uint32)
    return ((w >> np.uint32(9)).astype(np.float64) + 0.5) / 8388608.0


def gumbel_from_word(w) -> np.ndarray:
    return -np.log(-np.log(uniform_from_word(w)))


def uniforms(n: int, position: int, slot: int, seed: int) -> np.ndarray:
    """u_i in the open interval (0, 1), i = 0..n-1, as float64."""
    return uniform_from_word(words(n, position, slot, seed))


def gumbel(n: int, position: int, slot: int, seed: int) -> np.ndarray:
    return gumbel_from_word(words(n, position, slot, seed))


def sample_scores(logits: np.ndarray, temperature: float, position: int, slot: int, seed: int) -> np.ndarray:
    """z_i = logit_i / T + g_i (float64): the token is their argmax."""
    logits = np.asarray(logits, dtype=np.float64)
    return logits / temperature + gumbel(logits.shape[0], position, slot, seed)


def sample_token(logits: np.ndarray, temperature: float, position: int, slot: int, seed: int) -> int:
    """Greedy for temperature <= 0, else the Gumbel-max draw (lowest index on
    ties: np.argmax returns the first maximum)."""
    if temperature <= 0:
        return int(np.argmax(np.asarray(logits, dtype=np.float64)))
    return int(np.argmax(sample_scores(logits, temperature, position, slot, seed)))


# ---- top-k / top-p filtering ------------------------------------------------
#
# The filtered draw (the nucleus sampling of Holtzman, Buys, Du, Forbes,
# Choi, "The Curious Case of Neural Text Degeneration", ICLR 2020, with the
# usual top-k restriction before it):
#   1. candidates: the k largest logits, ordered by value descending and,
#      among equal values, by index ascending; k = top_k, or MAX_TOP_K when
#      only top_p is set (the nucleus is taken among the MAX_TOP_K most likely
#      tokens);
#   2. within the candidates, e_j = exp((z_j - z_max) / T) and S = sum of e_j;
#      keep the shortest prefix whose sum reaches top_p * S (at least one);
#   3. draw argmax_j(z_j / T + g_j) over the kept prefix, g_j the Gumbel noise
#      of vocabulary entry j as above (lowest index on ties).
# top_k = 0 and top_p = 1 is the unfiltered temperature draw.

MAX_TOP_K = 64


def candidates(logits: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest logits, by value descending then index ascending."""
    z = np.asarray(logits, dtype=np.float64)
    order = np.lexsort((np.arange(z.shape[0]), -z))  # last key is primary: -z, then index
    return order[:min(k, z.shape[0])]


def kept_set(logits: np.ndarray, temperature: float, top_k: int, top_p: float) -> np.ndarray:
    """The candidates a filtered draw chooses among, in candidate order."""
    z = np.asarray(logits, dtype=np.float64)
    if top_k <= 0 and top_p >= 1.0:
        return candidates(z, z.shape[0])
    k = top_k if top_k > 0 else MAX_TOP_K
    c = candidates(z, k)
    if top_p >= 1.0:
        return c
    e = np.exp((z[c] - z[c[0]]) / temperature)
    need = top_p * e.sum()
    acc, n = 0.0, 0
    while n < len(c):
        acc += e[n]
        n += 1
        if acc >= need:
            break
    return c[:n]


def sample_token_filtered(logits: np.ndarray, temperature: float, position: int, slot: int, seed: int,
                          top_k: int = 0, top_p: float = 1.0) -> int:
    """The filtered draw; greedy for temperature <= 0."""
    z = np.asarray(logits, dtype=np.float64)
    if temperature <= 0:
        return int(np.argmax(z))
    keep = kept_set(z, temperature, top_k, top_p)
    g = gumbel_from_word(words(z.shape[0], position, slot, seed))
    s = z[keep] / temperature + g[keep]
    best = np.flatnonzero(s == s.max())
    return int(keep[best].min())
