"""The learner with a per-row reference log-sum-exp (rz_loss_fwd_bwd_ref):
the kept terms are taken against the rollout's recorded log-sum-exp, so the
backward GEMMs use them directly (no dz pass).  Against the fp64 oracle on
the tiny workload, ragged mid-size shapes, masked tokens and peaked
softmaxes; against rz_loss_fwd_bwd (log pi, loss and D3 bitwise, dH and dW
to the rounding of one more bf16 step); the range flag when the reference
is far from the row's log-sum-exp; and the sharded form."""

import numpy as np
import pytest
import torch

import oracle
from invariant_logprobs_gb300 import shard, synth
from helpers import TOL_GRAD_REL_L2, TOL_LOGPI, bits, f64, rel_l2, scalar_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
PLAIN_VS_REF = 5e-3  # dH, dW of the two routes (each within 1e-2 of the oracle)


def _rand_bf16(shape, std, g):
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)


def _check(out, ref):
    assert np.max(np.abs(f64(out["logprob"]) - ref["logpi"])) <= TOL_LOGPI
    assert scalar_close(out["loss"].item(), ref["loss"]), (out["loss"].item(), ref["loss"])
    assert scalar_close(out["d3"].item(), ref["d3"]), (out["d3"].item(), ref["d3"])
    e_dH, e_dW = rel_l2(f64(out["dH"]), ref["dH"]), rel_l2(f64(out["dW"]), ref["dW"])
    assert e_dH <= TOL_GRAD_REL_L2 and e_dW <= TOL_GRAD_REL_L2, (e_dH, e_dW)


def _rollout(rz, H, W, tok):
    """log mu and the row's log-sum-exp as the rollout records them."""
    lse = torch.empty(H.shape[0], dtype=torch.float32, device=H.device)
    lm, lse = rz.rz_token_logprob(H, W, tok, lse_out=lse)
    return lm, lse


def _both(rz, H, W, tok, logmu, ref_lse, cu, adv, mask=None):
    """The reference route and the plain route on the same inputs."""
    assert isinstance(ref_lse, torch.Tensor)
    err = rz.new_err_flag(DEV)
    r = rz.rz_loss_fwd_bwd_ref(H, W, tok, logmu, ref_lse, cu, adv, err_flag=err,
                               action_mask=mask)
    p = rz.rz_loss_fwd_bwd(H, W, tok, logmu, cu, adv, action_mask=mask)
    torch.cuda.synchronize()
    assert err.item() == 0, err.item()
    assert np.array_equal(bits(r["logprob"]), bits(p["logprob"]))
    assert np.array_equal(bits(r["loss"]), bits(p["loss"]))
    assert np.array_equal(bits(r["d3"]), bits(p["d3"]))
    assert rel_l2(f64(r["dH"]), f64(p["dH"])) <= PLAIN_VS_REF
    assert rel_l2(f64(r["dW"]), f64(p["dW"])) <= PLAIN_VS_REF
    return r


def test_ref_tiny_vs_oracle(rz):
    b = synth.make_batch(synth.WORKLOADS["tiny"], device="cpu")
    tok = f64(b["tokens"])
    logmu, lse_mu = oracle.token_logprob(f64(b["H"]), f64(b["W_mu"]), tok)
    A = oracle.group_advantage(f64(b["rewards"]), b["G"]).astype(np.float32)
    lm = torch.tensor(logmu, dtype=torch.float32, device=DEV)
    R = torch.tensor(lse_mu, dtype=torch.float32, device=DEV)
    out = _both(rz, b["H"].to(DEV), b["W"].to(DEV), b["tokens"].to(DEV), lm, R, b["cu"].to(DEV),
                torch.tensor(A, device=DEV))
    ref = oracle.loss_fwd_bwd(f64(b["H"]), f64(b["W"]), tok, f64(lm), f64(b["cu"]),
                              A.astype(np.float64))
    _check(out, ref)


@pytest.mark.parametrize("T,d,V", [(1030, 136, 5000), (700, 512, 4099), (257, 2048, 1000)])
def test_ref_midsize_ragged_vs_oracle(rz, T, d, V):
    g = torch.Generator().manual_seed(T + d + V)
    H = _rand_bf16((T, d), 1.0, g)
    W = _rand_bf16((V, d), 0.05, g)
    W_mu = (W.float() + torch.randn(V, d, generator=g) * 0.002).to(torch.bfloat16)
    tok = torch.randint(0, V, (T,), generator=g, dtype=torch.int32)
    cuts = torch.sort(torch.randint(0, T + 1, (5,), generator=g)).values
    cu = torch.cat([torch.zeros(1, dtype=torch.int64), cuts, torch.full((1,), T, dtype=torch.int64)])
    adv = torch.randn(6, generator=g)
    lm, R = _rollout(rz, H.to(DEV), W_mu.to(DEV), tok.to(DEV))
    out = _both(rz, H.to(DEV), W.to(DEV), tok.to(DEV), lm, R, cu.to(DEV), adv.to(DEV))
    ref = oracle.loss_fwd_bwd(f64(H), f64(W), f64(tok), f64(lm), f64(cu), f64(adv))
    _check(out, ref)


def test_ref_masked_vs_oracle(rz):
    g = torch.Generator().manual_seed(11)
    T, d, V = 900, 256, 3000
    H = _rand_bf16((T, d), 1.0, g)
    W = _rand_bf16((V, d), 0.05, g)
    tok = torch.randint(0, V, (T,), generator=g, dtype=torch.int32)
    cu = torch.tensor([0, 200, 200, 650, T], dtype=torch.int64)
    adv = torch.tensor([0.5, -0.2, 1.0, -1.3])
    mask = (torch.rand(T, generator=g) < 0.7).to(torch.uint8)
    lm, R = _rollout(rz, H.to(DEV), W.to(DEV), tok.to(DEV))
    lm = lm + 0.05 * torch.randn(T, generator=g).to(DEV)
    out = _both(rz, H.to(DEV), W.to(DEV), tok.to(DEV), lm, R, cu.to(DEV), adv.to(DEV),
                mask.to(DEV))
    ref = oracle.loss_fwd_bwd(f64(H), f64(W), f64(tok), f64(lm), f64(cu), f64(adv),
                              mask=mask.numpy())
    _check(out, ref)
    # masked tokens get no gradient
    dH = out["dH"].float().cpu()
    assert float(dH[mask == 0].abs().max()) == 0.0


@pytest.mark.parametrize("std", [6.0, 14.0])
def test_ref_peaked_softmax_vs_oracle(rz, std):
    """Tokens drawn from their own peaked softmax: the sampled column's dz is
    c expm1(log pi) through the patched term; per-row parity for the rows
    with 1e-4 < 1 - p_a < 0.1."""
    g = torch.Generator().manual_seed(int(std) + 7)
    T, d, V = 700, 256, 4099
    H = _rand_bf16((T, d), 1.0, g)
    W = _rand_bf16((V, d), std / np.sqrt(d), g)
    z = H.double() @ W.double().T
    tok = torch.multinomial(torch.softmax(z, 1), 1, generator=g).squeeze(1).to(torch.int32)
    cu = torch.tensor([0, 150, 151, 400, T], dtype=torch.int64)
    # advantages that do not sum to zero: with a zero sum the loss is only the
    # small lag term and its relative error is that of w - 1
    adv = torch.tensor([0.7, -1.3, 0.4, 0.9])
    lm, R = _rollout(rz, H.to(DEV), W.to(DEV), tok.to(DEV))
    lm = lm + 0.05 * torch.randn(T, generator=g).to(DEV)
    out = _both(rz, H.to(DEV), W.to(DEV), tok.to(DEV), lm, R, cu.to(DEV), adv.to(DEV))
    ref = oracle.loss_fwd_bwd(f64(H), f64(W), f64(tok), f64(lm), f64(cu), f64(adv))
    _check(out, ref)
    gap = -np.expm1(ref["logpi"])
    rows = np.nonzero((gap > 1e-4) & (gap < 0.1))[0]
    assert len(rows) >= 20, len(rows)
    per_row = np.linalg.norm(f64(out["dH"])[rows] - ref["dH"][rows], axis=1) / \
        np.linalg.norm(ref["dH"][rows], axis=1)
    assert per_row.max() <= 2e-2, per_row.max()


def test_ref_far_from_the_rows_sets_the_range_flag(rz):
    g = torch.Generator().manual_seed(3)
    T, d, V = 300, 64, 2000
    H = _rand_bf16((T, d), 1.0, g).to(DEV)
    W = _rand_bf16((V, d), 0.1, g).to(DEV)
    tok = torch.randint(0, V, (T,), generator=g, dtype=torch.int32).to(DEV)
    cu = torch.tensor([0, 100, T], dtype=torch.int64, device=DEV)
    adv = torch.tensor([0.5, -0.5], device=DEV)
    lm, R = _rollout(rz, H, W, tok)
    for shift in (-100.0, 100.0):  # terms would overflow / the row factor would underflow
        err = rz.new_err_flag(DEV)
        out = rz.rz_loss_fwd_bwd_ref(H, W, tok, lm, R + shift, cu, adv, err_flag=err)
        torch.cuda.synchronize()
        assert err.item() & rz.RZ_DEVERR_RANGE
        # log pi, the loss and D3 do not depend on the reference
        assert out["d3"].item() == 0.0
    err = rz.new_err_flag(DEV)
    rz.rz_loss_fwd_bwd_ref(H, W, tok, lm, R + 30.0, cu, adv, err_flag=err)
    torch.cuda.synchronize()
    assert err.item() == 0  # 30 nats off is inside the range


def test_ref_two_chunks_and_zero_mismatch(rz):
    wl = synth.scaled(synth.WORKLOADS["qwen1p5b_lag2"], n_prompts=3, len_lo=300, len_hi=6000,
                      d=512, seed=79)
    b = synth.make_batch(wl, device=DEV)
    assert b["T"] > 38912
    lm, R = _rollout(rz, b["H"], b["W_mu"], b["tokens"])
    adv = rz.rz_group_advantage(b["rewards"], b["G"])
    _both(rz, b["H"], b["W"], b["tokens"], lm, R, b["cu"], adv)
    # at the rollout's own weights: w == 1, D3 == 0 exactly
    lm0, R0 = _rollout(rz, b["H"], b["W"], b["tokens"])
    out = rz.rz_loss_fwd_bwd_ref(b["H"], b["W"], b["tokens"], lm0, R0, b["cu"], adv)
    torch.cuda.synchronize()
    assert np.array_equal(bits(out["logprob"]), bits(lm0)) and out["d3"].item() == 0.0


def test_ref_sharded_equals_unsharded(rz):
    wl = synth.scaled(synth.WORKLOADS["qwen1p5b_lag2"], n_prompts=2, len_lo=300, len_hi=3000,
                      d=256, seed=81)
    b = synth.make_batch(wl, device=DEV)
    lm, R = _rollout(rz, b["H"], b["W_mu"], b["tokens"])
    adv = rz.rz_group_advantage(b["rewards"], b["G"])
    full = rz.rz_loss_fwd_bwd_ref(b["H"], b["W"], b["tokens"], lm, R, b["cu"], adv)
    cu = f64(b["cu"])
    dHs, parts = [], []
    for r0, r1 in shard.plan(cu, 3):
        t0, t1, cu_l = shard.local_batch(cu, (r0, r1))
        o = rz.rz_loss_fwd_bwd_shard(b["H"][t0:t1].contiguous(), b["W"],
                                     b["tokens"][t0:t1].contiguous(), lm[t0:t1].contiguous(),
                                     torch.as_tensor(cu_l, device=DEV), adv[r0:r1].contiguous(),
                                     b["B"], ref_lse=R[t0:t1].contiguous())
        dHs.append(o["dH"])
        parts.append(o["dW"])
    dW = rz.rz_sum_partials(torch.stack(parts))
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(dHs).view(torch.int16), full["dH"].view(torch.int16))
    assert rel_l2(f64(dW), f64(full["dW"])) <= 1e-4


@pytest.mark.parametrize("cuts,d,V,seed", [([0, 0, 3, 3, 10, 10], 200, 777, 5),
                                           ([0, 1], 64, 1000, 6)])
def test_ref_empty_responses_and_single_row(rz, cuts, d, V, seed):
    """Empty responses (first, middle and last) and a one-row batch on the
    reference route, against the oracle and the plain route."""
    g = torch.Generator().manual_seed(seed)
    T = cuts[-1]
    H = _rand_bf16((T, d), 1.0, g)
    W = _rand_bf16((V, d), 0.05, g)
    tok = torch.randint(0, V, (T,), generator=g, dtype=torch.int32)
    cu = torch.tensor(cuts, dtype=torch.int64)
    adv = torch.randn(len(cuts) - 1, generator=g)
    lm, R = _rollout(rz, H.to(DEV), W.to(DEV), tok.to(DEV))
    lm = lm + 0.05 * torch.randn(T, generator=g).to(DEV)
    out = _both(rz, H.to(DEV), W.to(DEV), tok.to(DEV), lm, R, cu.to(DEV), adv.to(DEV))
    ref = oracle.loss_fwd_bwd(f64(H), f64(W), f64(tok), f64(lm), f64(cu), f64(adv))
    _check(out, ref)


def test_ref_nan_reference_sets_the_range_flag(rz):
    g = torch.Generator().manual_seed(8)
    T, d, V = 200, 64, 1500
    H = _rand_bf16((T, d), 1.0, g).to(DEV)
    W = _rand_bf16((V, d), 0.1, g).to(DEV)
    tok = torch.randint(0, V, (T,), generator=g, dtype=torch.int32).to(DEV)
    cu = torch.tensor([0, 120, T], dtype=torch.int64, device=DEV)
    adv = torch.tensor([0.5, -0.5], device=DEV)
    lm, R = _rollout(rz, H, W, tok)
    R[37] = float("nan")
    err = rz.new_err_flag(DEV)
    rz.rz_loss_fwd_bwd_ref(H, W, tok, lm, R, cu, adv, err_flag=err)
    torch.cuda.synchronize()
    assert err.item() & rz.RZ_DEVERR_RANGE


@pytest.mark.parametrize("V", [1, 8, 264])
def test_ref_tiny_vocabularies(rz, V):
    """One-column, one-tile and ragged-tile vocabularies on the reference
    route: against the oracle and the plain route (V = 1: log pi = 0 and the
    gradients vanish)."""
    g = torch.Generator().manual_seed(V)
    T, d = 37, 64
    H = _rand_bf16((T, d), 1.0, g)
    W = _rand_bf16((V, d), 0.3, g)
    tok = torch.randint(0, V, (T,), generator=g, dtype=torch.int32)
    cu = torch.tensor([0, 20, T], dtype=torch.int64)
    adv = torch.tensor([0.8, -0.3])
    lm, R = _rollout(rz, H.to(DEV), W.to(DEV), tok.to(DEV))
    lm = lm - 0.02
    out = _both(rz, H.to(DEV), W.to(DEV), tok.to(DEV), lm, R, cu.to(DEV), adv.to(DEV))
    ref = oracle.loss_fwd_bwd(f64(H), f64(W), f64(tok), f64(lm), f64(cu), f64(adv))
    if V == 1:
        assert float(out["logprob"].abs().max()) == 0.0
        assert float(out["dH"].float().abs().max()) == 0.0
        assert float(out["dW"].abs().max()) == 0.0
    else:
        _check(out, ref)
