"""Property checks of the oracle over randomly drawn shapes (hypothesis):
identities that hold for any input, exactly or to fp64 rounding, so that a
mistake which a fixed example happens to hide still fails somewhere.

  * sum_a pi(a) = 1 and pi independent of a shift of a row's logits;
  * group advantages sum to 0 per group, unchanged by a per-group shift;
  * the loss is linear in A, invariant to permuting whole responses, and
    D3 >= 0; a masked token equals the token removed;
  * <dW, W> = <dH, H> (both are sum_t sum_v dz_tv z_tv); each column of dW
    sums to 0 over the vocabulary (each dz row does); one coordinate of dW
    and of dH against a central difference of the loss;
  * Score Centering: unchanged by a constant added to every advantage, and
    one coordinate of dW against a central difference of L_SC.
"""

import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402

SETTINGS = settings(max_examples=25, deadline=None, derandomize=True)


@st.composite
def problems(draw):
    seed = draw(st.integers(0, 2**31 - 1))
    rng = np.random.default_rng(seed)
    G = draw(st.sampled_from([1, 2, 3, 4]))
    B = G * draw(st.integers(1, 3))
    d = draw(st.integers(1, 6))
    V = draw(st.integers(1, 9))
    lengths = rng.integers(0, 5, B)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    T = int(cu[-1])
    H = rng.standard_normal((T, d))
    W = rng.standard_normal((V, d)) * draw(st.sampled_from([0.1, 1.0, 3.0]))
    tok = rng.integers(0, V, T)
    logmu = oracle.token_logprob(H, W + rng.standard_normal((V, d)) * 0.2, tok)[0]
    A = oracle.group_advantage(rng.random(B), G)
    mask = (rng.random(T) < 0.7).astype(np.uint8) if draw(st.booleans()) else None
    return dict(rng=rng, G=G, B=B, d=d, V=V, cu=cu, T=T, H=H, W=W, tok=tok, logmu=logmu, A=A,
                mask=mask)


@SETTINGS
@given(problems())
def test_policy_normalised_and_shift_invariant(p):
    if p["T"] == 0:
        return
    z = oracle.lmhead_logits(p["H"], p["W"])
    lse = oracle.logsumexp_rows(z)
    probs = np.exp(z - lse[:, None])
    assert np.allclose(probs.sum(1), 1.0, atol=1e-12)
    shift = p["rng"].standard_normal(p["T"])[:, None] * 50
    assert np.allclose(oracle.logsumexp_rows(z + shift) - shift[:, 0], lse, atol=1e-9)


@SETTINGS
@given(problems())
def test_group_advantage_centred_and_shift_invariant(p):
    rng = p["rng"]
    r = rng.random(p["B"])
    A = oracle.group_advantage(r, p["G"])
    assert np.allclose(A.reshape(-1, p["G"]).sum(1), 0.0, atol=1e-12)
    shift = np.repeat(rng.standard_normal(p["B"] // p["G"]), p["G"])
    assert np.allclose(oracle.group_advantage(r + shift, p["G"]), A, atol=1e-12)


@SETTINGS
@given(problems())
def test_loss_linear_permutation_invariant_d3_nonnegative(p):
    lp = oracle.token_logprob(p["H"], p["W"], p["tok"])[0]
    r1 = oracle.is_loss(lp, p["logmu"], p["cu"], p["A"], p["mask"])
    r2 = oracle.is_loss(lp, p["logmu"], p["cu"], 2.5 * p["A"], p["mask"])
    assert r2["loss"] == pytest.approx(2.5 * r1["loss"], rel=1e-12, abs=1e-15)
    assert r1["d3"] >= 0.0
    # permute whole responses
    B = p["B"]
    perm = p["rng"].permutation(B)
    cu = p["cu"]
    pieces = [np.arange(cu[i], cu[i + 1]) for i in perm]
    idx = np.concatenate(pieces) if pieces else np.zeros(0, np.int64)
    cu_p = np.concatenate([[0], np.cumsum([len(x) for x in pieces])]).astype(np.int64)
    m_p = None if p["mask"] is None else p["mask"][idx]
    r3 = oracle.is_loss(lp[idx], p["logmu"][idx], cu_p, p["A"][perm], m_p)
    assert r3["loss"] == pytest.approx(r1["loss"], rel=1e-12, abs=1e-15)
    assert r3["d3"] == pytest.approx(r1["d3"], rel=1e-12, abs=1e-15)


@SETTINGS
@given(problems())
def test_masked_token_equals_removed_token(p):
    if p["mask"] is None or p["T"] == 0:
        return
    keep = p["mask"] != 0
    lp = oracle.token_logprob(p["H"], p["W"], p["tok"])[0]
    full = oracle.is_loss(lp, p["logmu"], p["cu"], p["A"], p["mask"])
    seg = np.repeat(np.arange(p["B"]), np.diff(p["cu"]))  # response of each token
    counts = np.bincount(seg[keep], minlength=p["B"])
    cu_k = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    removed = oracle.is_loss(lp[keep], p["logmu"][keep], cu_k, p["A"])
    assert full["loss"] == pytest.approx(removed["loss"], rel=1e-12, abs=1e-15)
    assert full["d3"] == pytest.approx(removed["d3"], rel=1e-12, abs=1e-15)


@SETTINGS
@given(problems())
def test_gradient_identities_and_central_differences(p):
    H, W, tok, lm, cu, A, mask = p["H"], p["W"], p["tok"], p["logmu"], p["cu"], p["A"], p["mask"]
    r = oracle.loss_fwd_bwd(H, W, tok, lm, cu, A, mask=mask)
    dH, dW = r["dH"], r["dW"]
    scale = max(1.0, float(np.abs(dW).sum() * np.abs(W).sum()))
    assert abs(float((dW * W).sum()) - float((dH * H).sum())) <= 1e-12 * scale
    assert np.allclose(dW.sum(0), 0.0, atol=1e-12 * max(1.0, float(np.abs(dW).sum())))

    def loss_at(H2, W2):
        lp = oracle.token_logprob(H2, W2, tok)[0]
        return oracle.is_loss(lp, lm, cu, A, mask)["loss"]

    rng = p["rng"]
    h = 1e-6
    v, k = int(rng.integers(0, p["V"])), int(rng.integers(0, p["d"]))
    Wp, Wm = W.copy(), W.copy()
    Wp[v, k] += h
    Wm[v, k] -= h
    fd = (loss_at(H, Wp) - loss_at(H, Wm)) / (2 * h)
    assert fd == pytest.approx(dW[v, k], rel=1e-5, abs=1e-9)
    if p["T"] > 0:
        t = int(rng.integers(0, p["T"]))
        Hp, Hm = H.copy(), H.copy()
        Hp[t, k] += h
        Hm[t, k] -= h
        fd = (loss_at(Hp, W) - loss_at(Hm, W)) / (2 * h)
        assert fd == pytest.approx(dH[t, k], rel=1e-5, abs=1e-9)


@SETTINGS
@given(problems())
def test_score_centering_gradient_and_shift_invariance(p):
    H, W, tok, cu, A, mask = p["H"], p["W"], p["tok"], p["cu"], p["A"], p["mask"]
    r = oracle.sc_loss_fwd_bwd(H, W, tok, cu, A, mask=mask)
    # a constant added to every advantage changes neither loss nor gradient
    r2 = oracle.sc_loss_fwd_bwd(H, W, tok, cu, A + 0.75, mask=mask)
    assert r2["loss"] == pytest.approx(r["loss"], rel=1e-9, abs=1e-12)
    assert np.allclose(r2["dW"], r["dW"], atol=1e-12)
    assert np.allclose(r2["dH"], r["dH"], atol=1e-12)

    def loss_at(W2):
        lp = oracle.token_logprob(H, W2, tok)[0]
        return oracle.sc_loss(lp, cu, A, mask)["loss"]

    rng = p["rng"]
    h = 1e-6
    v, k = int(rng.integers(0, p["V"])), int(rng.integers(0, p["d"]))
    Wp, Wm = W.copy(), W.copy()
    Wp[v, k] += h
    Wm[v, k] -= h
    fd = (loss_at(Wp) - loss_at(Wm)) / (2 * h)
    assert fd == pytest.approx(r["dW"][v, k], rel=1e-5, abs=1e-9)
