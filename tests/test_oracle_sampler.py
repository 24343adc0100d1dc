"""Pins for the sampler oracle: the generator against its published
known-answer vectors, and the Gumbel-max rule against the closed-form
softmax probabilities it must reproduce."""

import math
import os

import numpy as np
import pytest
import scipy.stats

import oracle
from oracle import rz_sampler

KAT = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _kat():
    rows = []
    for line in open(KAT):
        if line.strip() and not line.startswith("#"):
            w = [int(x, 16) for x in line.split()]
            rows.append((w[0:4], w[4:6], w[6:10]))
    return rows


def test_philox_known_answers():
    rows = _kat()
    assert len(rows) == 3
    for ctr, key, want in rows:
        got = rz_sampler.philox4x32_10(np.array(ctr), np.array(key))
        assert [int(x) for x in got] == want


def test_uniforms_are_open_interval_and_23_bit():
    u = rz_sampler.uniforms(12345, 4096, seed=99)
    assert np.all(u > 0) and np.all(u < 1)
    assert np.all((u * 2 ** 23 - 0.5) == np.floor(u * 2 ** 23))


def test_gumbel_max_two_tokens_matches_softmax():
    # z = (0, log 3): softmax = (1/4, 3/4)
    H = np.ones((20000, 1))
    W = np.array([[0.0], [math.log(3.0)]])
    tok, lmu, _ = rz_sampler.sample_rows(H, W, np.arange(20000), seed=7)
    p1 = tok.mean()
    assert abs(p1 - 0.75) <= 4 * math.sqrt(0.75 * 0.25 / 20000)
    np.testing.assert_allclose(lmu[tok == 1], math.log(0.75), atol=1e-14)
    np.testing.assert_allclose(lmu[tok == 0], math.log(0.25), atol=1e-14)


def test_gumbel_max_three_tokens_matches_softmax():
    # z = (0, log 2, log 5): softmax = (1/8, 2/8, 5/8).  Unlike two tokens or
    # uniform logits, three unequal logits tell z + G from z - G apart
    # (z - G gives about (0.084, 0.245, 0.671)).
    n = 8000
    H = np.ones((n, 1))
    W = np.array([[0.0], [math.log(2.0)], [math.log(5.0)]])
    tok, _, _ = rz_sampler.sample_rows(H, W, np.arange(n) * 5 + 11, seed=23)
    counts = np.bincount(tok, minlength=3)
    p = scipy.stats.chisquare(counts, n * np.array([1.0, 2.0, 5.0]) / 8.0).pvalue
    assert p > 1e-4, counts


def test_gumbel_max_uniform_logits_chi_square():
    V, n = 16, 16000
    H = np.ones((n, 1))
    W = np.zeros((V, 1))
    tok, lmu, _ = rz_sampler.sample_rows(H, W, np.arange(n) + 10**12, seed=3)
    counts = np.bincount(tok, minlength=V)
    p = scipy.stats.chisquare(counts).pvalue
    assert p > 1e-4, counts
    np.testing.assert_allclose(lmu, -math.log(V), atol=1e-14)


def test_recorded_logmu_is_the_logprob_of_the_sampled_token():
    rng = np.random.default_rng(5)
    H = rng.standard_normal((40, 6))
    W = rng.standard_normal((30, 6))
    rid = rng.integers(0, 2**40, 40)
    tok, lmu, _ = rz_sampler.sample_rows(H, W, rid, seed=2**40 + 17)
    lp, _ = oracle.token_logprob(H, W, tok)
    np.testing.assert_allclose(lmu, lp, atol=1e-13)
    # a row's sample depends on its own row id only (not on its position)
    perm = rng.permutation(40)
    tok2, _, _ = rz_sampler.sample_rows(H[perm], W, rid[perm], seed=2**40 + 17)
    np.testing.assert_array_equal(tok2, tok[perm])


def test_key_of_at_the_zero_counter_uses_the_published_words():
    # row id 0 and seed 0 put tokens 0..3 at Philox counter (0, 0, 0, 0) under
    # key (0, 0): the first known-answer vector.  Their keys minus the logits
    # are the Gumbel draws -log(-log U) of those four published words.
    ctr, key, want = _kat()[0]
    assert ctr == [0, 0, 0, 0] and key == [0, 0]
    h = np.array([1.0, -2.0])
    W = np.array([[0.5, 0.0], [0.0, 1.0], [3.0, 1.0], [-1.0, -1.0], [2.0, 2.0]])
    keys, z = rz_sampler.key_of(h, W, 0, 0)
    np.testing.assert_array_equal(z, W @ h)
    u = np.array([((x >> 9) + 0.5) * 2.0 ** -23 for x in want])
    np.testing.assert_allclose(keys[:4] - z[:4], -np.log(-np.log(u)), rtol=0, atol=1e-12)


def test_key_of_agrees_with_the_sampled_rows():
    # row ids and a seed with both 32-bit halves non-zero: the token each row
    # draws holds the largest key that key_of gives for that row, and the
    # recorded margin is that key's lead over the runner-up
    rng = np.random.default_rng(11)
    H = rng.standard_normal((24, 5))
    W = rng.standard_normal((37, 5))
    rid = rng.integers(2**33, 2**62, 24)
    seed = (0x89ABCDEF << 32) | 0x01234567
    tok, _, margin = rz_sampler.sample_rows(H, W, rid, seed)
    for t in range(24):
        keys, z = rz_sampler.key_of(H[t], W, int(rid[t]), seed)
        np.testing.assert_allclose(z, oracle.lmhead_logits(H[t:t + 1], W)[0], atol=1e-12)
        assert int(np.argmax(keys)) == tok[t]
        srt = np.sort(keys)
        assert srt[-1] - srt[-2] == pytest.approx(margin[t], abs=1e-12)
    # another row id or seed draws other noise
    k0, _ = rz_sampler.key_of(H[0], W, int(rid[0]), seed)
    k1, _ = rz_sampler.key_of(H[0], W, int(rid[0]) + 1, seed)
    k2, _ = rz_sampler.key_of(H[0], W, int(rid[0]), seed ^ (1 << 40))
    assert not np.allclose(k0, k1) and not np.allclose(k0, k2)
