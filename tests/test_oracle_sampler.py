"""Pins for the sampler oracle: the generator against its published
known-answer vectors, and the two-level weighted reservoir against the
closed-form softmax probabilities it must reproduce."""

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
    x = rz_sampler.row_words(12345, np.arange(4096) * 977 + 3, 0, seed=99)
    u = rz_sampler.uniform_of(x.reshape(-1))
    assert np.all(u > 0) and np.all(u < 1)
    assert np.all((u * 2 ** 23 - 0.5) == np.floor(u * 2 ** 23))
    assert rz_sampler.uniform_of(0) == 2.0 ** -24
    assert rz_sampler.uniform_of(0xFFFFFFFF) == 1.0 - 2.0 ** -24


def test_draw_inside_one_chunk_uses_the_published_words():
    # row id 0 and seed 0: the first chunk's uniforms are words 0 and 1 of the
    # first known-answer vector (counter 0, key 0).  A one-chunk, one-segment
    # row always takes the chunk's draw, which visits columns 0,4,1,5,2,6,3,7
    # and stops where the running weight passes U2 * W.
    ctr, key, want = _kat()[0]
    assert ctr == [0, 0, 0, 0] and key == [0, 0]
    q = np.arange(1.0, 9.0)                      # weights 1..8 (z = log q)
    order = [0, 4, 1, 5, 2, 6, 3, 7]
    u2 = ((want[1] >> 9) + 0.5) * 2.0 ** -23
    cs = np.cumsum(q[order])
    expect = order[int(np.argmax(cs > u2 * q.sum()))]
    tok, lmu, _ = rz_sampler.sample_rows(np.ones((1, 1)), np.log(q)[:, None], [0], seed=0)
    assert tok[0] == expect
    assert lmu[0] == pytest.approx(math.log(q[expect] / q.sum()), abs=1e-14)
    np.testing.assert_array_equal(rz_sampler.draw_order(8), order)
    np.testing.assert_array_equal(rz_sampler.draw_order(6), [0, 4, 1, 5, 2, 3])


def test_segments_cover_the_vocabulary_in_whole_tiles():
    for V in (1, 8, 255, 256, 600, 4096, 16384, 16385, 151936):
        seg = rz_sampler.segments(V)
        assert seg[0][0] == 0 and seg[-1][1] == V
        assert all(seg[i][1] == seg[i + 1][0] for i in range(len(seg) - 1))
        assert len(seg) <= 64 and all(a % 256 == 0 for a, _ in seg)
    assert len(rz_sampler.segments(151936)) == 60
    assert rz_sampler.segments(600) == [(0, 256), (256, 512), (512, 600)]


def test_sampling_two_tokens_matches_softmax():
    # z = (0, log 3): softmax = (1/4, 3/4)
    H = np.ones((20000, 1))
    W = np.array([[0.0], [math.log(3.0)]])
    tok, lmu, _ = rz_sampler.sample_rows(H, W, np.arange(20000), seed=7)
    p1 = tok.mean()
    assert abs(p1 - 0.75) <= 4 * math.sqrt(0.75 * 0.25 / 20000)
    np.testing.assert_allclose(lmu[tok == 1], math.log(0.75), atol=1e-14)
    np.testing.assert_allclose(lmu[tok == 0], math.log(0.25), atol=1e-14)


def test_sampling_three_tokens_matches_softmax():
    # z = (0, log 2, log 5): softmax = (1/8, 2/8, 5/8)
    n = 8000
    H = np.ones((n, 1))
    W = np.array([[0.0], [math.log(2.0)], [math.log(5.0)]])
    tok, _, _ = rz_sampler.sample_rows(H, W, np.arange(n) * 5 + 11, seed=23)
    counts = np.bincount(tok, minlength=3)
    p = scipy.stats.chisquare(counts, n * np.array([1.0, 2.0, 5.0]) / 8.0).pvalue
    assert p > 1e-4, counts


def test_sampling_uniform_logits_chi_square():
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


def test_sampling_across_chunks_and_segments_matches_softmax():
    # V = 600: three segments (256, 256 and 88 columns) and 19 chunks, with
    # unequal masses per chunk, per class inside a chunk and per segment;
    # chi-square over every token
    V, n = 600, 60000
    v = np.arange(V)
    z = np.log1p(v % 7) + 0.6 * (v >= 256) - 0.4 * (v >= 512) + 0.3 * ((v // 32) % 3 == 1)
    H = np.ones((n, 1))
    tok, lmu, _ = rz_sampler.sample_rows(H, z[:, None], np.arange(n) * 13 + 7, seed=2**33 + 5)
    p = np.exp(z - z.max())
    p /= p.sum()
    counts = np.bincount(tok, minlength=V)
    assert scipy.stats.chisquare(counts, n * p).pvalue > 1e-4
    # per chunk and per segment as well (coarser bins, more power per bin)
    cb = np.bincount(tok // 32, minlength=19)
    assert scipy.stats.chisquare(cb, n * np.bincount(v // 32, weights=p)).pvalue > 1e-4
    np.testing.assert_allclose(lmu, np.log(p[tok]), atol=1e-12)
