"""Seeded sweep of random shapes through the learner and rollout entry
points against the oracle: T, d, V, response lengths (including empty
responses), group size and an optional action mask all vary, to catch edge
cases no hand-picked shape covers."""

import numpy as np
import pytest
import torch

import oracle
from helpers import (TOL_GRAD_REL_L2, TOL_LOGPI, f64, rel_l2, scalar_close)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(seed):
    rng = np.random.default_rng(seed)
    d = int(rng.integers(1, 97)) * 8                 # 8 .. 768
    V = int(rng.choice([rng.integers(1, 600), rng.integers(600, 6000)]))
    G = int(rng.choice([1, 2, 4, 8]))
    B = G * int(rng.integers(1, 5))
    lengths = rng.integers(0, 300, B)
    lengths[rng.random(B) < 0.15] = 0                # some empty responses
    if lengths.sum() == 0:
        lengths[0] = 1
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    T = int(cu[-1])
    g = torch.Generator().manual_seed(seed)
    H = torch.randn(T, d, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, d, generator=g) * (1.0 / np.sqrt(d))).to(torch.bfloat16)
    W_mu = (W.float() + torch.randn(V, d, generator=g) * 0.01).to(torch.bfloat16)
    tok = torch.randint(0, V, (T,), generator=g, dtype=torch.int32)
    rewards = torch.rand(B, generator=g)
    mask = (rng.random(T) < 0.8).astype(np.uint8) if rng.random() < 0.5 else None
    return dict(d=d, V=V, G=G, B=B, T=T, cu=cu, H=H, W=W, W_mu=W_mu, tok=tok,
                rewards=rewards, mask=mask)


@pytest.mark.parametrize("seed", list(range(12)))
def test_random_shape_learner_vs_oracle(rz, seed):
    c = _case(1000 + seed)
    Hd, Wd, tok = f64(c["H"]), f64(c["W"]), f64(c["tok"])
    logmu = oracle.token_logprob(Hd, f64(c["W_mu"]), tok)[0].astype(np.float32)
    A = oracle.group_advantage(f64(c["rewards"]), c["G"])
    A32 = A.astype(np.float32)  # the learner's input: the oracle's advantages at fp32
    adv_gpu = rz.rz_group_advantage(c["rewards"].to(DEV), c["G"])
    mask_t = None if c["mask"] is None else torch.tensor(c["mask"]).to(DEV)
    out = rz.rz_loss_fwd_bwd(c["H"].to(DEV), c["W"].to(DEV), c["tok"].to(DEV),
                             torch.tensor(logmu).to(DEV), torch.tensor(c["cu"]).to(DEV),
                             torch.tensor(A32).to(DEV), action_mask=mask_t)
    lp_roll, _ = rz.rz_token_logprob(c["H"].to(DEV), c["W"].to(DEV), c["tok"].to(DEV))
    torch.cuda.synchronize()
    np.testing.assert_allclose(f64(adv_gpu), A, atol=1e-6)
    ref = oracle.loss_fwd_bwd(Hd, Wd, tok, logmu.astype(np.float64), c["cu"],
                              A32.astype(np.float64), mask=c["mask"])
    assert np.max(np.abs(f64(out["logprob"]) - ref["logpi"])) <= TOL_LOGPI
    assert torch.equal(out["logprob"], lp_roll)
    assert scalar_close(out["loss"].item(), ref["loss"]), (out["loss"].item(), ref["loss"])
    assert scalar_close(out["d3"].item(), ref["d3"]), (out["d3"].item(), ref["d3"])
    for k in ("dH", "dW"):
        if np.linalg.norm(ref[k]) > 0:
            assert rel_l2(f64(out[k]), ref[k]) <= TOL_GRAD_REL_L2, k
        else:
            assert float(out[k].abs().max()) == 0.0
