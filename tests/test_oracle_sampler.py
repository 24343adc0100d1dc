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
