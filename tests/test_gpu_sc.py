"""Score Centering comparison estimator (rz_sc_loss_fwd_bwd) against the
fp64 oracle: log pi, the loss and dH, dW within the stated tolerances; log pi
bitwise the rollout's; for advantages that already sum to zero, bitwise the
IS learner at w = 1; invariant to a constant advantage shift."""

import numpy as np
import pytest
import torch

import oracle
from helpers import TOL_GRAD_REL_L2, TOL_LOGPI, TOL_SCALAR_REL, bits, f64, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _problem(T_lens, d, V, seed, w_scale=0.05):
    g = torch.Generator().manual_seed(seed)
    T = int(sum(T_lens))
    H = torch.randn(T, d, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, d, generator=g) * w_scale).to(torch.bfloat16)
    tok = torch.randint(0, V, (T,), generator=g, dtype=torch.int32)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(T_lens)]), dtype=torch.int64)
    adv = torch.randn(len(T_lens), generator=g) + 0.3
    return H, W, tok, cu, adv


def _loss_bound(got_lp, want_lp, cu, adv, mask):
    """|L_gpu - L| from the log pi errors alone: (1/B) sum_i |A_i - Abar| *
    max |delta log pi| (L is linear in log pi with those weights), plus the
    fp32 rounding of the reductions."""
    A = f64(adv)
    cu = f64(cu)
    valid = np.ones(len(got_lp), bool) if mask is None else f64(mask) != 0
    counts = np.array([valid[cu[i]:cu[i + 1]].sum() for i in range(len(A))])
    abar = A[counts > 0].mean()
    dlp = np.abs(f64(got_lp) - want_lp)[valid].max(initial=0.0)
    return np.abs(A - abar)[counts > 0].sum() / len(A) * dlp


@pytest.mark.parametrize("case", [
    dict(T_lens=[37, 0, 129, 300, 5, 258], d=256, V=5003, mask=True, seed=1),
    dict(T_lens=[64] * 8, d=136, V=777, mask=False, seed=2),
    dict(T_lens=[1000] * 40, d=64, V=1000, mask=True, seed=3),   # two 38,912-row chunks
])
def test_sc_matches_oracle(rz, case):
    H, W, tok, cu, adv = _problem(case["T_lens"], case["d"], case["V"], case["seed"])
    T = H.shape[0]
    mask = None
    if case["mask"]:
        g = torch.Generator().manual_seed(case["seed"] + 100)
        mask = (torch.rand(T, generator=g) > 0.25).to(torch.uint8)
    err = rz.new_err_flag(DEV)
    out = rz.rz_sc_loss_fwd_bwd(H.to(DEV), W.to(DEV), tok.to(DEV), cu.to(DEV), adv.to(DEV),
                                err_flag=err,
                                action_mask=None if mask is None else mask.to(DEV))
    torch.cuda.synchronize()
    assert err.item() == 0
    want = oracle.sc_loss_fwd_bwd(f64(H), f64(W), f64(tok), f64(cu), f64(adv),
                                  mask=None if mask is None else f64(mask))
    assert np.max(np.abs(f64(out["logprob"]) - want["logpi"])) <= TOL_LOGPI
    got = out["loss"].item()
    # against the exact loss: within what the log pi errors allow
    bound = _loss_bound(out["logprob"], want["logpi"], cu, adv, mask)
    assert abs(got - want["loss"]) <= bound + TOL_SCALAR_REL * abs(want["loss"]) + 1e-6
    assert rel_l2(f64(out["dH"]), want["dH"]) <= TOL_GRAD_REL_L2
    assert rel_l2(f64(out["dW"]), want["dW"]) <= TOL_GRAD_REL_L2
    if mask is not None:
        assert np.all(f64(out["dH"])[f64(mask) == 0] == 0.0)


def test_sc_bitwise_rollout_and_is_at_w_one(rz):
    # binary rewards, groups of 8: group-centred advantages sum to exactly 0,
    # so A - Abar == A and the SC coefficient equals the IS one at w = 1
    d, V = 256, 3001
    T_lens = [40, 33, 64, 7, 90, 12, 51, 23] * 2
    H, W, tok, cu, _ = _problem(T_lens, d, V, 7)
    g = torch.Generator().manual_seed(8)
    rewards = (torch.rand(len(T_lens), generator=g) > 0.5).float()
    Hd, Wd, td, cud = H.to(DEV), W.to(DEV), tok.to(DEV), cu.to(DEV)
    adv = rz.rz_group_advantage(rewards.to(DEV), 8)
    lp, _ = rz.rz_token_logprob(Hd, Wd, td)
    sc = rz.rz_sc_loss_fwd_bwd(Hd, Wd, td, cud, adv)
    isl = rz.rz_loss_fwd_bwd(Hd, Wd, td, lp, cud, adv)
    torch.cuda.synchronize()
    assert float(adv.double().sum()) == 0.0
    assert np.array_equal(bits(sc["logprob"]), bits(lp))
    assert isl["d3"].item() == 0.0
    assert torch.equal(sc["dH"], isl["dH"])
    assert torch.equal(sc["dW"], isl["dW"])


def test_sc_advantage_shift_invariance(rz):
    H, W, tok, cu, adv = _problem([50, 0, 77, 130, 21], 128, 2048, 9)
    Hd, Wd, td, cud = H.to(DEV), W.to(DEV), tok.to(DEV), cu.to(DEV)
    a = rz.rz_sc_loss_fwd_bwd(Hd, Wd, td, cud, adv.to(DEV))
    b = rz.rz_sc_loss_fwd_bwd(Hd, Wd, td, cud, (adv + 3.25).to(DEV))
    torch.cuda.synchronize()
    # the centred advantages agree to fp32 rounding, so only bf16 rounding
    # flips of dz separate the two; without centring they would differ by O(1)
    assert rel_l2(f64(b["dW"]), f64(a["dW"])) <= 1e-3
    assert rel_l2(f64(b["dH"]), f64(a["dH"])) <= 1e-3
    assert abs(b["loss"].item() - a["loss"].item()) <= 1e-5 * abs(a["loss"].item()) + 1e-5


def test_sc_empty_batch(rz):
    d, V = 64, 512
    W = torch.randn(V, d, device=DEV).to(torch.bfloat16)
    H0 = torch.empty(0, d, dtype=torch.bfloat16, device=DEV)
    t0 = torch.empty(0, dtype=torch.int32, device=DEV)
    cu = torch.zeros(3, dtype=torch.int64, device=DEV)
    dW = torch.full((V, d), 7.0, device=DEV)
    out = rz.rz_sc_loss_fwd_bwd(H0, W, t0, cu, torch.tensor([0.5, -0.25], device=DEV), dW=dW)
    torch.cuda.synchronize()
    assert out["loss"].item() == 0.0
    assert bool(torch.all(out["dW"] == 0))
