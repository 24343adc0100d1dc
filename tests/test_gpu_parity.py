"""GPU-vs-oracle parity through the C ABI (small and mid sizes, ragged tails,
several tiles), plus the tensor-core GEMM against a plain fp32 matmul."""

import numpy as np
import pytest
import torch

import oracle
from invariant_logprobs_gb300 import synth
from helpers import (TOL_GRAD_REL_L2, TOL_LOGPI, f64, rel_l2, scalar_close)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _rand_bf16(shape, std, g):
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)


@pytest.mark.parametrize("T,d,V", [(300, 256, 1000), (1, 64, 256), (129, 2048, 513),
                                   (520, 1536, 4096), (257, 136, 300)])
def test_lmhead_logits_matches_fp32_matmul(rz, T, d, V):
    g = torch.Generator().manual_seed(T * 7 + d + V)
    H = _rand_bf16((T, d), 1.0, g)
    W = _rand_bf16((V, d), 0.05, g)
    z = rz.rz_lmhead_logits(H.to(DEV), W.to(DEV))
    torch.cuda.synchronize()
    ref = H.double() @ W.double().T
    err = (z.cpu().double() - ref).abs().max().item()
    scale = (H.double().abs() @ W.double().abs().T).max().item()
    assert err <= 1e-5 * scale, (err, scale)


def _tiny_inputs(wl, device="cpu"):
    b = synth.make_batch(wl, device=device)
    logmu64, _ = oracle.token_logprob(f64(b["H"]), f64(b["W_mu"]), f64(b["tokens"]))
    b["logmu"] = torch.tensor(logmu64, dtype=torch.float32)
    b["adv"] = torch.tensor(oracle.group_advantage(f64(b["rewards"]), b["G"]),
                            dtype=torch.float32)
    return b


def _run_learner(rz, b):
    out = rz.rz_loss_fwd_bwd(b["H"].to(DEV), b["W"].to(DEV), b["tokens"].to(DEV),
                             b["logmu"].to(DEV), b["cu"].to(DEV), b["adv"].to(DEV))
    torch.cuda.synchronize()
    return out


def _check_learner(out, ref):
    lp = f64(out["logprob"])
    assert np.max(np.abs(lp - ref["logpi"])) <= TOL_LOGPI
    loss = float(out["loss"].item())
    d3 = float(out["d3"].item())
    assert scalar_close(loss, ref["loss"]), (loss, ref["loss"])
    assert scalar_close(d3, ref["d3"]), (d3, ref["d3"])
    e_dh = rel_l2(f64(out["dH"]), ref["dH"])
    e_dw = rel_l2(f64(out["dW"]), ref["dW"])
    assert e_dh <= TOL_GRAD_REL_L2, e_dh
    assert e_dw <= TOL_GRAD_REL_L2, e_dw
    return e_dh, e_dw


def test_token_logprob_tiny_vs_oracle(rz):
    b = _tiny_inputs(synth.WORKLOADS["tiny"])
    lp, lse = rz.rz_token_logprob(b["H"].to(DEV), b["W"].to(DEV), b["tokens"].to(DEV),
                                  lse_out=torch.empty(b["T"], device=DEV))
    torch.cuda.synchronize()
    ref_lp, ref_lse = oracle.token_logprob(f64(b["H"]), f64(b["W"]), f64(b["tokens"]))
    assert np.max(np.abs(f64(lp) - ref_lp)) <= TOL_LOGPI
    assert np.max(np.abs(f64(lse) - ref_lse)) <= TOL_LOGPI
    # much tighter in practice: fp32 accumulation of exact bf16 products
    assert np.max(np.abs(f64(lp) - ref_lp)) <= 1e-4


@pytest.mark.parametrize("V", [1024, 151936, 1000])
def test_zero_weights_give_minus_log_v(rz, V):
    T, d = 77, 64
    H = torch.randn(T, d).to(torch.bfloat16).to(DEV)
    W = torch.zeros(V, d, dtype=torch.bfloat16, device=DEV)
    tok = torch.randint(0, V, (T,), dtype=torch.int32, device=DEV)
    lp, _ = rz.rz_token_logprob(H, W, tok)
    want = np.float32(-np.log(V))
    got = lp.cpu().numpy()
    ulp = np.spacing(np.abs(want))
    assert np.all(np.abs(got - want) <= 2 * ulp), (got[:4], want)


def test_learner_tiny_vs_oracle(rz):
    b = _tiny_inputs(synth.WORKLOADS["tiny"])
    out = _run_learner(rz, b)
    ref = oracle.loss_fwd_bwd(f64(b["H"]), f64(b["W"]), f64(b["tokens"]), f64(b["logmu"]),
                              f64(b["cu"]), f64(b["adv"]))
    _check_learner(out, ref)


@pytest.mark.parametrize("shape", [
    dict(n_prompts=3, group=4, len_lo=1, len_hi=200, d=512, V=5000),      # ragged V tail
    dict(n_prompts=2, group=8, len_lo=60, len_hi=90, d=1536, V=2304),     # d = 6 N-tiles
    dict(n_prompts=1, group=5, len_lo=0, len_hi=40, d=200, V=777),        # empty responses, d % 64
])
def test_learner_midsize_vs_oracle(rz, shape):
    wl = synth.Workload("mid", shape["n_prompts"], shape["group"], shape["len_lo"],
                        shape["len_hi"], shape["d"], shape["V"], "bernoulli", 0.5, "uniform",
                        4, 2e-3, 4242)
    b = _tiny_inputs(wl)
    out = _run_learner(rz, b)
    ref = oracle.loss_fwd_bwd(f64(b["H"]), f64(b["W"]), f64(b["tokens"]), f64(b["logmu"]),
                              f64(b["cu"]), f64(b["adv"]))
    _check_learner(out, ref)


def test_learner_multi_chunk_vs_oracle(rz):
    # more rows than one backward chunk (38912): exercises chunked dz and the
    # fixed-order dW accumulation over chunks.
    wl = synth.Workload("chunks", 1, 3, 15000, 16000, 64, 384, "uniform", 0.0, "uniform",
                        4, 3e-2, 777)
    b = _tiny_inputs(wl)
    assert b["T"] > 38912
    out = _run_learner(rz, b)
    ref = oracle.loss_fwd_bwd(f64(b["H"]), f64(b["W"]), f64(b["tokens"]), f64(b["logmu"]),
                              f64(b["cu"]), f64(b["adv"]))
    _check_learner(out, ref)


def test_group_advantage_vs_oracle(rz):
    g = torch.Generator().manual_seed(5)
    for B, G, kind in [(256, 8, "bern"), (128, 8, "unif"), (12, 3, "unif"), (7, 1, "unif")]:
        r = (torch.rand(B, generator=g) < 0.4).float() if kind == "bern" else torch.rand(B, generator=g)
        A = rz.rz_group_advantage(r.to(DEV), G)
        torch.cuda.synchronize()
        ref = oracle.group_advantage(f64(r), G)
        np.testing.assert_allclose(f64(A), ref, atol=1e-7)
        if kind == "bern" and G in (1, 2, 4, 8):
            assert np.all(f64(A).reshape(-1, G).sum(1) == 0.0)


@pytest.mark.parametrize("T,B,spread", [(1_114_112, 128, 0.08), (5000, 256, 1.5), (3, 2, 0.0)])
def test_is_loss_and_d3_vs_oracle(rz, T, B, spread):
    g = torch.Generator().manual_seed(T + B)
    cuts = torch.sort(torch.randint(0, T + 1, (B - 1,), generator=g)).values
    cu = torch.cat([torch.zeros(1, dtype=torch.int64), cuts, torch.full((1,), T, dtype=torch.int64)])
    logpi = -torch.rand(T, generator=g) * 12
    logmu = logpi + torch.randn(T, generator=g) * spread
    adv = torch.randn(B, generator=g)
    loss, d3, coef = rz.rz_is_loss(logpi.to(DEV), logmu.to(DEV), cu.to(DEV), adv.to(DEV),
                                   coef_out=torch.empty(T, device=DEV))
    d3b = rz.rz_d3(logpi.to(DEV), logmu.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.is_loss(f64(logpi), f64(logmu), f64(cu), f64(adv))
    assert scalar_close(loss.item(), ref["loss"]), (loss.item(), ref["loss"])
    assert scalar_close(d3.item(), ref["d3"]), (d3.item(), ref["d3"])
    assert scalar_close(d3b.item(), ref["d3"]), (d3b.item(), ref["d3"])
    np.testing.assert_allclose(f64(coef), ref["c"], rtol=1e-5, atol=1e-12)


@pytest.mark.parametrize("T,V,B", [(600, 1024, 6), (1030, 151936, 4), (5, 8, 5)])
def test_logits_variant_vs_oracle(rz, T, V, B):
    g = torch.Generator().manual_seed(T + V)
    logits = (torch.randn(T, V, generator=g) * 3.0).to(torch.bfloat16)
    tok = torch.randint(0, V, (T,), generator=g, dtype=torch.int32)
    cu = torch.linspace(0, T, B + 1).round().to(torch.int64)
    adv = torch.randn(B, generator=g)
    lp64 = oracle.logits_loss_fwd_bwd(f64(logits), f64(tok), np.zeros(T), f64(cu), f64(adv))["logpi"]
    logmu = torch.tensor(lp64, dtype=torch.float32) + torch.randn(T, generator=g) * 0.05
    rows = np.unique(np.concatenate([np.arange(min(T, 8)), np.random.default_rng(0).integers(0, T, 32)]))
    ref = oracle.logits_loss_fwd_bwd(f64(logits), f64(tok), f64(logmu), f64(cu), f64(adv), rows=rows)
    buf = logits.to(DEV)
    out = rz.rz_logits_loss_fwd_bwd(buf, tok.to(DEV), logmu.to(DEV), cu.to(DEV), adv.to(DEV))
    torch.cuda.synchronize()
    assert np.max(np.abs(f64(out["logprob"]) - ref["logpi"])) <= TOL_LOGPI
    assert scalar_close(out["loss"].item(), ref["loss"]), (out["loss"].item(), ref["loss"])
    assert scalar_close(out["d3"].item(), ref["d3"]), (out["d3"].item(), ref["d3"])
    dz = f64(buf[torch.as_tensor(rows, device=DEV)])
    assert rel_l2(dz, ref["dz"]) <= TOL_GRAD_REL_L2


@pytest.mark.parametrize("T,spread", [(1_114_112, 0.08), (777, 2.0), (1, 0.3)])
def test_is_stats_vs_oracle(rz, T, spread):
    g = torch.Generator().manual_seed(T)
    logpi = -torch.rand(T, generator=g) * 12
    logmu = logpi + torch.randn(T, generator=g) * spread
    st = rz.rz_is_stats(logpi.to(DEV), logmu.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.is_stats(f64(logpi), f64(logmu))
    got = dict(zip(rz.IS_STATS_FIELDS, st.cpu().double().tolist()))
    for k in ("d3", "k1", "k2", "w_mean"):
        assert scalar_close(got[k], ref[k]), (k, got[k], ref[k])
    for k in ("w_max", "w_min", "absd_max"):
        assert abs(got[k] - ref[k]) <= 1e-6 * max(1.0, abs(ref[k])), (k, got[k], ref[k])
    # D3 of the diagnostics equals rz_d3 bit for bit? (different reduction
    # layouts are allowed to differ by rounding; both must match the oracle)
    d3b = rz.rz_d3(logpi.to(DEV), logmu.to(DEV)).item()
    assert scalar_close(d3b, got["d3"])


def _mask_for(cu, T, seed, frac=0.7):
    rng = np.random.default_rng(seed)
    m = (rng.random(T) < frac).astype(np.uint8)
    if len(cu) > 3:
        m[int(cu[1]):int(cu[2])] = 0   # one response without any action token
    return m


def test_learner_masked_vs_oracle(rz):
    wl = synth.Workload("masked", 3, 4, 1, 180, 512, 5000, "bernoulli", 0.5, "uniform",
                        4, 2e-3, 4343)
    b = _tiny_inputs(wl)
    cu = f64(b["cu"])
    mask = _mask_for(cu, b["T"], 1)
    out = rz.rz_loss_fwd_bwd(b["H"].to(DEV), b["W"].to(DEV), b["tokens"].to(DEV),
                             b["logmu"].to(DEV), b["cu"].to(DEV), b["adv"].to(DEV),
                             action_mask=torch.tensor(mask).to(DEV))
    torch.cuda.synchronize()
    ref = oracle.loss_fwd_bwd(f64(b["H"]), f64(b["W"]), f64(b["tokens"]), f64(b["logmu"]),
                              cu, f64(b["adv"]), mask=mask)
    _check_learner(out, ref)
    assert bool(torch.all(out["dH"][torch.tensor(mask == 0).to(DEV)] == 0))


@pytest.mark.parametrize("T,B", [(1_114_112, 128), (997, 9)])
def test_is_loss_masked_vs_oracle(rz, T, B):
    g = torch.Generator().manual_seed(T * 3 + B)
    cuts = torch.sort(torch.randint(0, T + 1, (B - 1,), generator=g)).values
    cu = torch.cat([torch.zeros(1, dtype=torch.int64), cuts, torch.full((1,), T, dtype=torch.int64)])
    logpi = -torch.rand(T, generator=g) * 12
    logmu = logpi + torch.randn(T, generator=g) * 0.1
    adv = torch.randn(B, generator=g)
    mask = _mask_for(f64(cu), T, 2)
    loss, d3, coef = rz.rz_is_loss(logpi.to(DEV), logmu.to(DEV), cu.to(DEV), adv.to(DEV),
                                   coef_out=torch.empty(T, device=DEV),
                                   action_mask=torch.tensor(mask).to(DEV))
    torch.cuda.synchronize()
    ref = oracle.is_loss(f64(logpi), f64(logmu), f64(cu), f64(adv), mask=mask)
    assert scalar_close(loss.item(), ref["loss"]), (loss.item(), ref["loss"])
    assert scalar_close(d3.item(), ref["d3"]), (d3.item(), ref["d3"])
    np.testing.assert_allclose(f64(coef), ref["c"], rtol=1e-5, atol=1e-12)


def test_logits_variant_masked_vs_oracle(rz):
    T, V, B = 700, 2048, 7
    g = torch.Generator().manual_seed(77)
    logits = (torch.randn(T, V, generator=g) * 3.0).to(torch.bfloat16)
    tok = torch.randint(0, V, (T,), generator=g, dtype=torch.int32)
    cu = torch.linspace(0, T, B + 1).round().to(torch.int64)
    adv = torch.randn(B, generator=g)
    logmu = torch.randn(T, generator=g) * 0.05 - 8.0
    mask = _mask_for(f64(cu), T, 3)
    ref = oracle.logits_loss_fwd_bwd(f64(logits), f64(tok), f64(logmu), f64(cu), f64(adv),
                                     mask=mask)
    buf = logits.to(DEV)
    out = rz.rz_logits_loss_fwd_bwd(buf, tok.to(DEV), logmu.to(DEV), cu.to(DEV), adv.to(DEV),
                                    action_mask=torch.tensor(mask).to(DEV))
    torch.cuda.synchronize()
    assert np.max(np.abs(f64(out["logprob"]) - ref["logpi"])) <= TOL_LOGPI
    assert scalar_close(out["loss"].item(), ref["loss"]), (out["loss"].item(), ref["loss"])
    assert scalar_close(out["d3"].item(), ref["d3"]), (out["d3"].item(), ref["d3"])
    assert rel_l2(f64(buf), ref["dz"]) <= TOL_GRAD_REL_L2
    assert bool(torch.all(buf[torch.tensor(mask == 0).to(DEV)] == 0))


@pytest.mark.parametrize("T,d,V", [(5, 8, 37), (64, 4096, 1000)])
def test_learner_extreme_d(rz, T, d, V):
    wl = synth.Workload("extreme_d", 1, 2, T // 2, T // 2, d, V, "uniform", 0.0, "uniform",
                        4, 1e-2, 55 + d)
    b = _tiny_inputs(wl)
    out = _run_learner(rz, b)
    ref = oracle.loss_fwd_bwd(f64(b["H"]), f64(b["W"]), f64(b["tokens"]), f64(b["logmu"]),
                              f64(b["cu"]), f64(b["adv"]))
    _check_learner(out, ref)


def test_single_token_vocabulary(rz):
    # V = 1: softmax is 1, log pi = 0 exactly, dz = c (1 - 1) = 0
    T, d = 40, 64
    H = torch.randn(T, d).to(torch.bfloat16).to(DEV)
    W = torch.randn(1, d).to(torch.bfloat16).to(DEV)
    tok = torch.zeros(T, dtype=torch.int32, device=DEV)
    cu = torch.tensor([0, 15, 40], dtype=torch.int64, device=DEV)
    adv = torch.tensor([1.0, -1.0], device=DEV)
    logmu = torch.full((T,), -0.5, device=DEV)
    out = rz.rz_loss_fwd_bwd(H, W, tok, logmu, cu, adv)
    torch.cuda.synchronize()
    assert bool(torch.all(out["logprob"] == 0.0))
    assert bool(torch.all(out["dH"] == 0)) and bool(torch.all(out["dW"] == 0))
    ref = oracle.is_loss(np.zeros(T), np.full(T, -0.5), f64(cu), f64(adv))
    assert scalar_close(out["loss"].item(), ref["loss"])
    assert scalar_close(out["d3"].item(), ref["d3"])


@pytest.mark.parametrize("T", [38912, 38913])
def test_learner_chunk_boundary(rz, T):
    # exactly one backward chunk, and one row into a second chunk
    g = torch.Generator().manual_seed(T)
    d, V, B = 64, 256, 4
    H = torch.randn(T, d, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, d, generator=g) * 0.1).to(torch.bfloat16)
    tok = torch.randint(0, V, (T,), generator=g, dtype=torch.int32)
    cu = torch.tensor([0, 1000, 20000, T - 1, T], dtype=torch.int64)
    adv = torch.tensor([0.3, -0.2, 0.5, -0.6])
    lm = torch.tensor(oracle.token_logprob(f64(H), f64(W), f64(tok))[0], dtype=torch.float32)
    lm = lm + torch.randn(T, generator=g) * 0.05
    out = rz.rz_loss_fwd_bwd(H.to(DEV), W.to(DEV), tok.to(DEV), lm.to(DEV), cu.to(DEV), adv.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.loss_fwd_bwd(f64(H), f64(W), f64(tok), f64(lm), f64(cu), f64(adv))
    _check_learner(out, ref)


def test_equal_rewards_give_zero_advantage_loss_and_gradients(rz):
    # a group whose rewards are all equal has A = 0: no loss, no gradient
    wl = synth.Workload("flat", 1, 6, 20, 50, 128, 700, "uniform", 0.0, "uniform", 4, 1e-2, 9)
    b = _tiny_inputs(wl)
    r = torch.full((6,), 0.37)
    adv = rz.rz_group_advantage(r.to(DEV), 6)
    out = rz.rz_loss_fwd_bwd(b["H"].to(DEV), b["W"].to(DEV), b["tokens"].to(DEV),
                             b["logmu"].to(DEV), b["cu"].to(DEV), adv)
    torch.cuda.synchronize()
    assert bool(torch.all(adv == 0))
    assert out["loss"].item() == 0.0
    assert bool(torch.all(out["dH"] == 0)) and bool(torch.all(out["dW"] == 0))


@pytest.mark.parametrize("std", [6.0, 14.0])
def test_learner_peaked_softmax_vs_oracle(rz, std):
    """Peaked rows (logit standard deviation 6 and 14, tokens drawn from the
    softmax itself): most terms of a row are many orders below the row's
    maximum and the sampled token's probability is often close to 1, where
    dz_a = c (p_a - 1) must keep its digits.  Whole-batch parity, and per
    row for the rows with 1e-4 < 1 - p_a < 0.1."""
    g = torch.Generator().manual_seed(int(std))
    T, d, V = 700, 256, 4099
    H = _rand_bf16((T, d), 1.0, g)
    W = _rand_bf16((V, d), std / np.sqrt(d), g)
    z = H.double() @ W.double().T
    tok = torch.multinomial(torch.softmax(z, 1), 1, generator=g).squeeze(1).to(torch.int32)
    cu = torch.tensor([0, 150, 151, 400, 700], dtype=torch.int64)
    adv = torch.tensor([0.7, -1.3, 0.4, 0.2])
    lp64, _ = oracle.token_logprob(f64(H), f64(W), f64(tok))
    logmu = torch.tensor(lp64 + np.random.default_rng(int(std)).normal(0, 0.05, T),
                         dtype=torch.float32)
    out = rz.rz_loss_fwd_bwd(H.to(DEV), W.to(DEV), tok.to(DEV), logmu.to(DEV), cu.to(DEV),
                             adv.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.loss_fwd_bwd(f64(H), f64(W), f64(tok), f64(logmu), f64(cu), f64(adv))
    _check_learner(out, ref)
    gap = -np.expm1(ref["logpi"])                        # 1 - p_a
    rows = np.nonzero((gap > 1e-4) & (gap < 0.1))[0]
    assert len(rows) >= 20, len(rows)
    got = f64(out["dH"])[rows]
    want = ref["dH"][rows]
    per_row = np.linalg.norm(got - want, axis=1) / np.linalg.norm(want, axis=1)
    assert per_row.max() <= 2e-2, per_row.max()


@pytest.mark.parametrize("std", [6.0, 14.0])
def test_logits_variant_peaked_softmax_vs_oracle(rz, std):
    """Given logits with standard deviation 6 and 14 and tokens drawn from
    their own softmax: the sampled token's probability is often close to 1,
    where log pi is near 0 and dz_a = c (p_a - 1) must keep its digits (the
    kernel forms c expm1(log pi) there).  Whole-batch parity, and per row for
    the rows with 1e-4 < 1 - p_a < 0.1."""
    g = torch.Generator().manual_seed(int(std) + 100)
    T, V, B = 1200, 151936, 6
    logits = (torch.randn(T, V, generator=g) * std).to(torch.bfloat16)
    tok = torch.multinomial(torch.softmax(logits.double(), 1), 1, generator=g)
    tok = tok.squeeze(1).to(torch.int32)
    cu = torch.linspace(0, T, B + 1).round().to(torch.int64)
    adv = torch.randn(B, generator=g)
    lp64 = oracle.logits_loss_fwd_bwd(f64(logits), f64(tok), np.zeros(T), f64(cu), f64(adv),
                                      rows=np.zeros(0, np.int64))["logpi"]
    logmu = torch.tensor(lp64, dtype=torch.float32) + torch.randn(T, generator=g) * 0.05
    ref = oracle.logits_loss_fwd_bwd(f64(logits), f64(tok), f64(logmu), f64(cu), f64(adv))
    buf = logits.to(DEV)
    out = rz.rz_logits_loss_fwd_bwd(buf, tok.to(DEV), logmu.to(DEV), cu.to(DEV), adv.to(DEV))
    torch.cuda.synchronize()
    assert np.max(np.abs(f64(out["logprob"]) - ref["logpi"])) <= TOL_LOGPI
    assert scalar_close(out["loss"].item(), ref["loss"]), (out["loss"].item(), ref["loss"])
    assert scalar_close(out["d3"].item(), ref["d3"]), (out["d3"].item(), ref["d3"])
    dz = f64(buf)
    assert rel_l2(dz, ref["dz"]) <= TOL_GRAD_REL_L2
    gap = -np.expm1(ref["logpi"])                        # 1 - p_a
    rows = np.nonzero((gap > 1e-4) & (gap < 0.1))[0]
    assert len(rows) >= 20, len(rows)
    per_row = np.linalg.norm(dz[rows] - ref["dz"][rows], axis=1) / \
        np.linalg.norm(ref["dz"][rows], axis=1)
    assert per_row.max() <= 2e-2, per_row.max()
    # the sampled column itself, where the old p - 1 form lost its digits
    a_got = dz[rows, f64(tok)[rows]]
    a_want = ref["dz"][rows, f64(tok)[rows]]
    assert np.max(np.abs(a_got - a_want) / np.abs(a_want)) <= 2e-2


def test_logits_variant_large_vocabulary(rz):
    """A 262,144-column row (512 KB of bf16): the row kernel's shared-memory
    stash holds an eighth of it and the second pass re-reads the rest."""
    T, V, B = 70, 262144, 2
    g = torch.Generator().manual_seed(5)
    logits = (torch.randn(T, V, generator=g) * 3.0).to(torch.bfloat16)
    tok = torch.randint(0, V, (T,), generator=g, dtype=torch.int32)
    cu = torch.tensor([0, 33, T], dtype=torch.int64)
    adv = torch.tensor([0.6, -0.6])
    lp64 = oracle.logits_loss_fwd_bwd(f64(logits), f64(tok), np.zeros(T), f64(cu), f64(adv),
                                      rows=np.zeros(0, np.int64))["logpi"]
    logmu = torch.tensor(lp64, dtype=torch.float32) + torch.randn(T, generator=g) * 0.05
    ref = oracle.logits_loss_fwd_bwd(f64(logits), f64(tok), f64(logmu), f64(cu), f64(adv))
    buf = logits.to(DEV)
    out = rz.rz_logits_loss_fwd_bwd(buf, tok.to(DEV), logmu.to(DEV), cu.to(DEV), adv.to(DEV))
    torch.cuda.synchronize()
    assert np.max(np.abs(f64(out["logprob"]) - ref["logpi"])) <= TOL_LOGPI
    assert scalar_close(out["loss"].item(), ref["loss"])
    assert scalar_close(out["d3"].item(), ref["d3"])
    assert rel_l2(f64(buf), ref["dz"]) <= TOL_GRAD_REL_L2
