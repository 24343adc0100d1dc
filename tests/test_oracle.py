"""Pins for the CPU oracle: each checks it against something other than
itself (hand-worked examples, closed forms, library routines, finite
differences, autograd, enumeration identities), so that a dropped term, a
wrong sign or a transposed operand fails at least one of them."""

import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.txt")
_SAFE = {"log": math.log, "exp": math.exp, "sqrt": math.sqrt, "pi": math.pi}


def _load_golden():
    blocks, cur = {}, None
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("["):
                cur = blocks.setdefault(line.strip("[]"), {})
                continue
            k, v = [x.strip() for x in line.split("=", 1)]
            if k == "cite":
                cur[k] = v
            else:
                cur[k] = np.array([eval(t, {"__builtins__": {}}, _SAFE)
                                   for t in v.split()], dtype=np.float64)
    return blocks


GOLD = _load_golden()


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- worked examples

def test_golden_blocks_have_citations():
    assert GOLD and all("cite" in b for b in GOLD.values())


def test_golden_loss_two_responses():
    g = GOLD["loss_two_responses"]
    r = oracle.is_loss(g["logpi"], g["logmu"], g["cu_seqlens"].astype(np.int64),
                       g["adv"])
    assert r["loss"] == pytest.approx(g["loss"][0], abs=1e-15)
    assert r["d3"] == pytest.approx(g["d3"][0], abs=1e-15)
    np.testing.assert_allclose(r["c"], g["c"], atol=1e-15)
    assert oracle.d3(g["logpi"], g["logmu"]) == pytest.approx(g["d3"][0], abs=1e-15)


def test_golden_advantage():
    g = GOLD["advantage_two_groups"]
    A = oracle.group_advantage(g["rewards"], int(g["G"][0]))
    np.testing.assert_array_equal(A, g["adv"])


def test_golden_logprob_three_tokens():
    g = GOLD["logprob_three_tokens"]
    H = g["H"].reshape(1, 2)
    W = g["W"].reshape(3, 2)
    for a in range(3):
        lp, _ = oracle.token_logprob(H, W, np.array([a]))
        assert lp[0] == pytest.approx(g["logpi_all"][a], abs=1e-15)


def test_golden_zero_weights_exact():
    g = GOLD["zero_weights"]
    rng = _rng(0)
    for V, want in zip(g["V"].astype(int), g["logpi"]):
        H = rng.standard_normal((5, 8))
        W = np.zeros((V, 8))
        lp, _ = oracle.token_logprob(H, W, rng.integers(0, V, 5))
        assert np.all(lp == want)  # exact: z = 0, sum = V, log V


def test_golden_gradient_uniform():
    g = GOLD["gradient_uniform_two_tokens"]
    H = g["H"].reshape(1, 1)
    W = g["W"].reshape(2, 1)
    tok = g["token"].astype(np.int64)
    lp, _ = oracle.token_logprob(H, W, tok)
    r = oracle.loss_fwd_bwd(H, W, tok, lp, np.array([0, 1]), g["adv"])
    assert r["loss"] == pytest.approx(g["loss"][0], abs=1e-15)
    np.testing.assert_allclose(r["dH"].ravel(), g["dH"], atol=1e-15)
    np.testing.assert_allclose(r["dW"].ravel(), g["dW"], atol=1e-15)


# ---------------------------------------------------------------- log pi

def test_logprob_matches_scipy_log_softmax_bruteforce():
    rng = _rng(1)
    T, d, V = 7, 5, 11
    H = rng.standard_normal((T, d))
    W = rng.standard_normal((V, d))
    tok = rng.integers(0, V, T)
    lp, lse = oracle.token_logprob(H, W, tok)
    # logits by explicit loops (no matmul), normaliser by scipy
    z = np.array([[sum(H[t, k] * W[v, k] for k in range(d)) for v in range(V)]
                  for t in range(T)])
    ref = scipy.special.log_softmax(z, axis=1)[np.arange(T), tok]
    np.testing.assert_allclose(lp, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(z, axis=1), atol=1e-12)


def test_logprob_v2_is_log_sigmoid():
    rng = _rng(2)
    H = rng.standard_normal((50, 3)) * 4
    W = rng.standard_normal((2, 3))
    tok = rng.integers(0, 2, 50)
    lp, _ = oracle.token_logprob(H, W, tok)
    z = H @ W.T
    other = 1 - tok
    ref = scipy.special.log_expit(z[np.arange(50), tok] - z[np.arange(50), other])
    np.testing.assert_allclose(lp, ref, atol=1e-12)


def test_logprob_shift_invariance_and_large_logits():
    rng = _rng(3)
    H = rng.standard_normal((6, 4))
    W = rng.standard_normal((9, 4))
    tok = rng.integers(0, 9, 6)
    lp, _ = oracle.token_logprob(H, W, tok)
    # append a hidden unit equal to 1 whose weight is the same for every
    # vocab row: adds a per-row constant (here 1000, past the largest
    # argument of a finite fp64 exp, ~709) to all logits, so only a
    # log-sum-exp taken relative to the row maximum stays finite.
    H2 = np.concatenate([H, np.ones((6, 1))], 1)
    W2 = np.concatenate([W, np.full((9, 1), 1000.0)], 1)
    lp2, lse2 = oracle.token_logprob(H2, W2, tok)
    np.testing.assert_allclose(lp2, lp, atol=1e-10)
    assert np.all(np.isfinite(lse2))


def test_logprob_probabilities_sum_to_one():
    rng = _rng(4)
    H = rng.standard_normal((3, 6))
    W = rng.standard_normal((13, 6))
    for t in range(3):
        lps = [oracle.token_logprob(H[t:t + 1], W, np.array([a]))[0][0]
               for a in range(13)]
        assert math.fsum(math.exp(x) for x in lps) == pytest.approx(1.0, abs=1e-14)


def test_rows_subset_equals_full():
    rng = _rng(5)
    H = rng.standard_normal((40, 6))
    W = rng.standard_normal((30, 6))
    tok = rng.integers(0, 30, 40)
    lp, lse = oracle.token_logprob(H, W, tok)
    rows = np.array([39, 0, 17, 17, 3])
    lpr, lser = oracle.token_logprob_rows(H, W, tok, rows)
    np.testing.assert_array_equal(lpr, lp[rows])
    np.testing.assert_array_equal(lser, lse[rows])


# ---------------------------------------------------------------- advantages

def test_advantage_group_sums_zero_and_shift_invariance():
    rng = _rng(6)
    r = rng.random(64)
    A = oracle.group_advantage(r, 8)
    np.testing.assert_allclose(A.reshape(8, 8).sum(1), 0, atol=1e-14)
    shift = np.repeat(rng.standard_normal(8) * 10, 8)
    np.testing.assert_allclose(oracle.group_advantage(r + shift, 8), A, atol=1e-12)
    # binary rewards with G a power of two: exact zero sums
    rb = (rng.random(64) < 0.4).astype(np.float64)
    assert np.all(oracle.group_advantage(rb, 8).reshape(8, 8).sum(1) == 0.0)


def test_advantage_degenerate_groups():
    r = np.array([0.3, 0.9, 0.1])
    np.testing.assert_array_equal(oracle.group_advantage(r, 1), 0.0)
    np.testing.assert_allclose(oracle.group_advantage(r, 3), r - r.mean())
    with pytest.raises(ValueError):
        oracle.group_advantage(r, 2)


# ---------------------------------------------------------------- loss and D3

def _ragged(rng, B, lo, hi):
    L = rng.integers(lo, hi + 1, B)
    return np.concatenate([[0], np.cumsum(L)]).astype(np.int64)


def test_loss_at_w_one_is_minus_mean_advantage_and_d3_zero():
    rng = _rng(7)
    cu = _ragged(rng, 12, 1, 9)
    T = int(cu[-1])
    lp = -rng.random(T) * 10
    A = rng.standard_normal(12)
    r = oracle.is_loss(lp, lp, cu, A)
    assert r["d3"] == 0.0
    assert r["loss"] == pytest.approx(-A.mean(), abs=1e-14)


def test_loss_linear_in_advantage_and_permutation_invariant():
    rng = _rng(8)
    cu = _ragged(rng, 10, 1, 7)
    T = int(cu[-1])
    lp = -rng.random(T) * 5
    lm = lp + rng.standard_normal(T) * 0.3
    A1, A2 = rng.standard_normal(10), rng.standard_normal(10)
    L1 = oracle.is_loss(lp, lm, cu, A1)["loss"]
    L2 = oracle.is_loss(lp, lm, cu, A2)["loss"]
    L12 = oracle.is_loss(lp, lm, cu, 2 * A1 - 3 * A2)["loss"]
    assert L12 == pytest.approx(2 * L1 - 3 * L2, abs=1e-12)
    # permute whole responses
    perm = rng.permutation(10)
    segs = [np.arange(cu[i], cu[i + 1]) for i in range(10)]
    idx = np.concatenate([segs[i] for i in perm])
    cu_p = np.concatenate([[0], np.cumsum([len(segs[i]) for i in perm])])
    Lp = oracle.is_loss(lp[idx], lm[idx], cu_p, A1[perm])["loss"]
    assert Lp == pytest.approx(L1, abs=1e-12)


def test_loss_empty_response_counts_in_B_only():
    lp = np.array([-1.0, -2.0])
    lm = np.array([-1.5, -2.0])
    A = np.array([1.0, 5.0])
    r_a = oracle.is_loss(lp, lm, np.array([0, 2, 2]), A)
    w = np.exp(lp - lm)
    assert r_a["loss"] == pytest.approx(-(1.0 * w.mean()) / 2, abs=1e-15)


def test_d3_nonnegative_small_gap_and_closed_form():
    rng = _rng(9)
    d = rng.standard_normal(1000) * 2
    lp = -rng.random(1000) * 5
    assert oracle.d3(lp, lp - d) >= 0
    small = rng.standard_normal(1000) * 1e-3
    assert oracle.d3(lp, lp - small) == pytest.approx(np.mean(small ** 2 / 2), rel=2e-3)
    # single token with w = e: D3 = e - 2
    assert oracle.d3(np.array([1.0]), np.array([0.0])) == pytest.approx(math.e - 2, abs=1e-15)
    assert oracle.d3(np.array([]), np.array([])) == 0.0


# ---------------------------------------------------------------- gradients

def _tiny_problem(seed, T_lo=1, T_hi=4, B=3, d=4, V=6, w_scale=0.7):
    rng = _rng(seed)
    cu = _ragged(rng, B, T_lo, T_hi)
    T = int(cu[-1])
    H = rng.standard_normal((T, d))
    W = rng.standard_normal((V, d)) * w_scale
    tok = rng.integers(0, V, T)
    lm = oracle.token_logprob(H, W + rng.standard_normal((V, d)) * 0.2, tok)[0]
    A = rng.standard_normal(B)
    return H, W, tok, lm, cu, A


def test_gradients_match_central_differences():
    H, W, tok, lm, cu, A = _tiny_problem(10)
    r = oracle.loss_fwd_bwd(H, W, tok, lm, cu, A)

    def L(Hx, Wx):
        return oracle.loss_fwd_bwd(Hx, Wx, tok, lm, cu, A)["loss"]

    eps = 1e-6
    gH = np.zeros_like(H)
    for idx in np.ndindex(H.shape):
        Hp, Hm = H.copy(), H.copy()
        Hp[idx] += eps
        Hm[idx] -= eps
        gH[idx] = (L(Hp, W) - L(Hm, W)) / (2 * eps)
    gW = np.zeros_like(W)
    for idx in np.ndindex(W.shape):
        Wp, Wm = W.copy(), W.copy()
        Wp[idx] += eps
        Wm[idx] -= eps
        gW[idx] = (L(H, Wp) - L(H, Wm)) / (2 * eps)
    assert np.linalg.norm(r["dH"] - gH) <= 1e-6 * np.linalg.norm(gH)
    assert np.linalg.norm(r["dW"] - gW) <= 1e-6 * np.linalg.norm(gW)


def test_gradients_match_torch_autograd():
    H, W, tok, lm, cu, A = _tiny_problem(11, T_lo=2, T_hi=9, B=5, d=7, V=13)
    r = oracle.loss_fwd_bwd(H, W, tok, lm, cu, A)
    Ht = torch.tensor(H, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    logp = torch.log_softmax(Ht @ Wt.T, dim=1)[torch.arange(len(tok)), torch.tensor(tok)]
    w = torch.exp(logp - torch.tensor(lm))
    B = len(A)
    loss = 0
    for i in range(B):
        s, e = int(cu[i]), int(cu[i + 1])
        if e > s:
            loss = loss + float(A[i]) * w[s:e].mean()
    loss = -loss / B
    loss.backward()
    assert float(loss.detach()) == pytest.approx(r["loss"], abs=1e-13)
    np.testing.assert_allclose(r["dH"], Ht.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(r["dW"], Wt.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(r["logpi"], logp.detach().numpy(), atol=1e-12)


def test_gradient_at_w_one_is_plain_reinforce():
    # log mu := log pi (w = 1).  The gradient must equal the gradient of the
    # textbook surrogate -(1/B) sum_i (A_i/T_i) sum_t log pi (torch autograd).
    H, W, tok, _, cu, A = _tiny_problem(12, T_lo=1, T_hi=6, B=4, d=5, V=8)
    lp, _ = oracle.token_logprob(H, W, tok)
    r = oracle.loss_fwd_bwd(H, W, tok, lp, cu, A)
    Ht = torch.tensor(H, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    logp = torch.log_softmax(Ht @ Wt.T, 1)[torch.arange(len(tok)), torch.tensor(tok)]
    sur = 0
    for i in range(len(A)):
        s, e = int(cu[i]), int(cu[i + 1])
        sur = sur + float(A[i]) * logp[s:e].mean()
    (-sur / len(A)).backward()
    np.testing.assert_allclose(r["dH"], Ht.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(r["dW"], Wt.grad.numpy(), atol=1e-12)


def test_gradient_zero_weights_closed_form():
    rng = _rng(13)
    T, d, V = 9, 4, 5
    H = rng.standard_normal((T, d))
    W = np.zeros((V, d))
    tok = rng.integers(0, V, T)
    lm = -np.log(V) + rng.standard_normal(T) * 0.1
    cu = np.array([0, 4, 9])
    A = np.array([0.7, -0.7])
    r = oracle.loss_fwd_bwd(H, W, tok, lm, cu, A)
    assert np.all(r["dH"] == 0.0)
    w = np.exp(-np.log(V) - lm)
    Ti = np.array([4] * 4 + [5] * 5)
    Ai = np.array([0.7] * 4 + [-0.7] * 5)
    c = Ai * w / (2 * Ti)
    want = np.zeros((V, d))
    for t in range(T):
        for v in range(V):
            want[v] += c[t] * ((1.0 / V) - (1.0 if tok[t] == v else 0.0)) * H[t]
    np.testing.assert_allclose(r["dW"], want, atol=1e-14)


def test_is_identities_by_enumeration():
    """E_{a~mu}[w(a) dz(a)] over all V tokens: with a constant advantage it is
    zero (E_q[w s] = 0); with a token-dependent advantage it equals the exact
    policy gradient -grad_z E_{a~pi}[A(a)] (g_IS = g*)."""
    rng = _rng(14)
    d, V = 3, 7
    h = rng.standard_normal((1, d))
    W = rng.standard_normal((V, d))
    Wmu = W + rng.standard_normal((V, d)) * 0.5
    logmu_all = np.array([oracle.token_logprob(h, Wmu, np.array([a]))[0][0]
                          for a in range(V)])
    mu = np.exp(logmu_all)
    cu = np.array([0, 1])
    acc_const = np.zeros((V, d))
    Avals = rng.standard_normal(V)
    acc_var = np.zeros((V, d))
    for a in range(V):
        lm = logmu_all[a:a + 1]
        r1 = oracle.loss_fwd_bwd(h, W, np.array([a]), lm, cu, np.array([1.0]))
        acc_const += mu[a] * r1["dW"]
        r2 = oracle.loss_fwd_bwd(h, W, np.array([a]), lm, cu, Avals[a:a + 1])
        acc_var += mu[a] * r2["dW"]
    np.testing.assert_allclose(acc_const, 0.0, atol=1e-14)
    Wt = torch.tensor(W, requires_grad=True)
    p = torch.softmax(torch.tensor(h) @ Wt.T, 1)[0]
    (p * torch.tensor(Avals)).sum().backward()
    np.testing.assert_allclose(acc_var, -Wt.grad.numpy(), atol=1e-13)


def test_logits_variant_matches_hidden_variant():
    H, W, tok, lm, cu, A = _tiny_problem(15, T_lo=2, T_hi=5, B=4, d=6, V=9)
    r = oracle.loss_fwd_bwd(H, W, tok, lm, cu, A)
    z = H @ W.T
    rl = oracle.logits_loss_fwd_bwd(z, tok, lm, cu, A)
    assert rl["loss"] == pytest.approx(r["loss"], abs=1e-14)
    assert rl["d3"] == pytest.approx(r["d3"], abs=1e-14)
    np.testing.assert_allclose(rl["dz"] @ W, r["dH"], atol=1e-13)
    np.testing.assert_allclose(rl["dz"].T @ H, r["dW"], atol=1e-13)
    # dz rows sum to zero (softmax minus one-hot)
    np.testing.assert_allclose(rl["dz"].sum(1), 0.0, atol=1e-14)
    sub = oracle.logits_loss_fwd_bwd(z, tok, lm, cu, A, rows=np.array([3, 0]))
    np.testing.assert_array_equal(sub["dz"], rl["dz"][[3, 0]])


def test_log_gap_decomposition_zero_kernel_term():
    """log pi_k - log mu_v = (log pi_k - log pi_v) + (log pi_v - log mu_v):
    when the rollout's recorded logprob is computed by the same definition at
    the same weights, the second term is exactly zero and D3 = 0."""
    rng = _rng(16)
    H = rng.standard_normal((20, 5))
    Wv = rng.standard_normal((11, 5))
    tok = rng.integers(0, 11, 20)
    mu_v = oracle.token_logprob(H, Wv, tok)[0]
    pi_v = oracle.token_logprob(H, Wv, tok)[0]
    assert np.all(pi_v - mu_v == 0.0)
    assert oracle.d3(pi_v, mu_v) == 0.0


# ---------------------------------------------------------------- diagnostics

def test_is_stats_closed_forms():
    lp = np.array([-3.0, -5.0, -1.0])
    r = oracle.is_stats(lp, lp - 0.25)            # d = 0.25 everywhere
    assert r["k1"] == pytest.approx(-0.25, abs=1e-15)
    assert r["k2"] == pytest.approx(0.03125, abs=1e-15)
    assert r["d3"] == pytest.approx(math.exp(0.25) - 1.25, abs=1e-15)
    assert r["w_max"] == r["w_min"] == pytest.approx(math.exp(0.25))
    assert r["absd_max"] == pytest.approx(0.25)
    z = oracle.is_stats(np.array([]), np.array([]))
    assert all(v == 0.0 for v in z.values())


def test_kl_estimators_by_enumeration():
    """Weighting tokens by mu instead of sampling them: both k1 and k3 (= D3
    per token) have expectation KL(mu || pi) (scipy rel_entr)."""
    rng = _rng(21)
    V = 9
    pi = rng.random(V); pi /= pi.sum()
    mu = rng.random(V); mu /= mu.sum()
    kl = float(np.sum(scipy.special.rel_entr(mu, pi)))
    lp, lm = np.log(pi), np.log(mu)
    k1 = sum(mu[a] * oracle.is_stats(lp[a:a + 1], lm[a:a + 1])["k1"] for a in range(V))
    k3 = sum(mu[a] * oracle.is_stats(lp[a:a + 1], lm[a:a + 1])["d3"] for a in range(V))
    assert k1 == pytest.approx(kl, abs=1e-14)
    assert k3 == pytest.approx(kl, abs=1e-14)


def test_peak_to_median():
    assert oracle.peak_to_median([1.0, 2.0, 3.0, 100.0]) == pytest.approx(40.0)
    assert oracle.peak_to_median([2.0, 2.0, 2.0]) == 1.0
    assert oracle.peak_to_median([3.0, 1.0, 2.0]) == pytest.approx(1.5)


# ---------------------------------------------------------------- action masks

def test_mask_all_ones_is_no_mask():
    H, W, tok, lm, cu, A = _tiny_problem(30, T_lo=1, T_hi=7, B=5, d=4, V=9)
    r0 = oracle.loss_fwd_bwd(H, W, tok, lm, cu, A)
    r1 = oracle.loss_fwd_bwd(H, W, tok, lm, cu, A, mask=np.ones(len(tok), dtype=np.uint8))
    for k in ("loss", "d3"):
        assert r1[k] == r0[k]
    np.testing.assert_array_equal(r1["dW"], r0["dW"])


def test_masked_tokens_equal_removed_tokens():
    """Masking a token out must give exactly the loss, D3 and dW of the batch
    with that token removed, and a zero dH row for it."""
    H, W, tok, lm, cu, A = _tiny_problem(31, T_lo=2, T_hi=8, B=6, d=5, V=11)
    rng = _rng(32)
    T = len(tok)
    mask = (rng.random(T) < 0.7).astype(np.uint8)
    mask[cu[2]:cu[3]] = 0                        # one response fully masked
    rm = oracle.loss_fwd_bwd(H, W, tok, lm, cu, A, mask=mask)
    keep = mask != 0
    lengths = [int(keep[cu[i]:cu[i + 1]].sum()) for i in range(len(A))]
    cu_k = np.concatenate([[0], np.cumsum(lengths)])
    rk = oracle.loss_fwd_bwd(H[keep], W, tok[keep], lm[keep], cu_k, A)
    assert rm["loss"] == pytest.approx(rk["loss"], abs=1e-14)
    assert rm["d3"] == pytest.approx(rk["d3"], abs=1e-14)
    np.testing.assert_allclose(rm["dW"], rk["dW"], atol=1e-14)
    np.testing.assert_allclose(rm["dH"][keep], rk["dH"], atol=1e-14)
    assert np.all(rm["dH"][~keep] == 0.0)
    assert np.all(rm["c"][~keep] == 0.0)


# ---------------------------------------------------------------- score centering

def _scores(H, W, tok):
    """Per-token score s_t = grad_(H, W) log pi_t by autograd: list of
    (dH_t, dW_t) arrays."""
    out = []
    for t in range(len(tok)):
        Ht = torch.tensor(H, requires_grad=True)
        Wt = torch.tensor(W, requires_grad=True)
        lp = torch.log_softmax(Ht @ Wt.T, 1)[t, int(tok[t])]
        lp.backward()
        out.append((Ht.grad.numpy().copy(), Wt.grad.numpy().copy()))
    return out


def test_sc_gradient_is_the_literal_centred_score_update():
    """-(dH, dW) of L_SC equals (1/B) sum_i (A_i/T_i) sum_t (s_t - sbar),
    sbar the mean per-token-averaged score over responses with tokens,
    assembled from autograd scores (with a masked token and an empty
    response in the batch)."""
    H, W, tok, _, cu, A = _tiny_problem(40, T_lo=1, T_hi=5, B=5, d=4, V=7)
    T = len(tok)
    mask = np.ones(T, dtype=np.uint8)
    mask[cu[1]:cu[2]] = 0          # response 1 has no valid token
    mask[cu[3]] = 0                # one masked token in response 3
    r = oracle.sc_loss_fwd_bwd(H, W, tok, cu, A, mask=mask)
    sc = _scores(H, W, tok)
    B = len(A)
    resp_mean = []
    for i in range(B):
        ts = [t for t in range(cu[i], cu[i + 1]) if mask[t]]
        if ts:
            resp_mean.append((i, sum(sc[t][0] for t in ts) / len(ts),
                              sum(sc[t][1] for t in ts) / len(ts)))
    sbar_H = sum(m[1] for m in resp_mean) / len(resp_mean)
    sbar_W = sum(m[2] for m in resp_mean) / len(resp_mean)
    gH = sum(A[i] * (mH - sbar_H) for i, mH, _ in resp_mean) / B
    gW = sum(A[i] * (mW - sbar_W) for i, _, mW in resp_mean) / B
    np.testing.assert_allclose(-r["dH"], gH, atol=1e-13)
    np.testing.assert_allclose(-r["dW"], gW, atol=1e-13)


def test_sc_gradient_matches_central_differences():
    H, W, tok, _, cu, A = _tiny_problem(41)
    r = oracle.sc_loss_fwd_bwd(H, W, tok, cu, A)
    eps = 1e-6
    gW = np.zeros_like(W)
    for idx in np.ndindex(W.shape):
        Wp, Wm = W.copy(), W.copy()
        Wp[idx] += eps
        Wm[idx] -= eps
        gW[idx] = (oracle.sc_loss_fwd_bwd(H, Wp, tok, cu, A)["loss"] -
                   oracle.sc_loss_fwd_bwd(H, Wm, tok, cu, A)["loss"]) / (2 * eps)
    assert np.linalg.norm(r["dW"] - gW) <= 1e-6 * np.linalg.norm(gW)


def test_sc_invariant_to_advantage_shift_and_reduces_to_reinforce():
    H, W, tok, _, cu, A = _tiny_problem(42, T_lo=0, T_hi=6, B=6, d=5, V=8)
    r = oracle.sc_loss_fwd_bwd(H, W, tok, cu, A)
    r2 = oracle.sc_loss_fwd_bwd(H, W, tok, cu, A + 3.25)
    np.testing.assert_allclose(r2["dH"], r["dH"], atol=1e-13)
    np.testing.assert_allclose(r2["dW"], r["dW"], atol=1e-13)
    # advantages already centred over the responses with tokens: SC is the
    # IS update at w = 1 (log mu := log pi), i.e. plain REINFORCE
    counts = np.diff(cu)
    Ac = A - A[counts > 0].mean()
    rs = oracle.sc_loss_fwd_bwd(H, W, tok, cu, Ac)
    lp, _ = oracle.token_logprob(H, W, tok)
    ri = oracle.loss_fwd_bwd(H, W, tok, lp, cu, Ac)
    assert abs(rs["abar"]) < 1e-15
    np.testing.assert_allclose(rs["dH"], ri["dH"], atol=1e-13)
    np.testing.assert_allclose(rs["dW"], ri["dW"], atol=1e-13)
    np.testing.assert_allclose(rs["dW"], r["dW"], atol=1e-13)


def test_sc_expectation_is_sampler_covariance_by_enumeration():
    """Score centering keeps Cov_q(A, s) [item 03]: over every pair of
    one-token responses drawn i.i.d. from q at the same state (B = 2), the
    exact expectation of the SC update is (1 - 1/B) Cov_q(A, s), the usual
    finite-batch factor of a batch-mean baseline; the uncentred update
    E_q[A s] differs from it by the drift E_q[A] E_q[s] (item 02)."""
    rng = _rng(43)
    d, V = 3, 5
    h = rng.standard_normal((1, d))
    W = rng.standard_normal((V, d))
    Wq = W + rng.standard_normal((V, d)) * 0.6
    q = np.exp(np.array([oracle.token_logprob(h, Wq, np.array([a]))[0][0] for a in range(V)]))
    Aof = rng.standard_normal(V) + 0.8     # E_q[A] != 0: there is a drift to remove
    s = [_scores(h, W, np.array([a]))[0][1] for a in range(V)]   # dlog pi(a)/dW
    cov = sum(q[a] * Aof[a] * s[a] for a in range(V)) - \
        sum(q * Aof) * sum(q[a] * s[a] for a in range(V))
    exp_g = np.zeros_like(W)
    H2 = np.vstack([h, h])
    for a1 in range(V):
        for a2 in range(V):
            r = oracle.sc_loss_fwd_bwd(H2, W, np.array([a1, a2]), np.array([0, 1, 2]),
                                       np.array([Aof[a1], Aof[a2]]))
            exp_g += q[a1] * q[a2] * (-r["dW"])
    np.testing.assert_allclose(exp_g, 0.5 * cov, atol=1e-13)
    drift = sum(q * Aof) * sum(q[a] * s[a] for a in range(V))
    assert np.linalg.norm(drift) > 1e-2
