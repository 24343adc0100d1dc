"""Full-size parity at the benchmark's shapes and launch configuration
(1.5B-shaped lag-2 and 4B-shaped lag-64 learner batches, ~1.1M tokens,
V = 151936), checked on sampled rows the oracle computes one by one and on
identities that hold at any size:

  * log pi of 64 sampled rows vs the oracle;
  * dH of the sampled rows vs the oracle's dz_t W (dz from the oracle's own
    softmax of the row, the recorded log mu, A_i, B and T_i);
  * <dW, W> == <dH, H> (both equal sum_t sum_v dz_tv z_tv), tying dW to the
    row-checked dH;
  * the loss/D3 of the fused call equal rz_is_loss on its own log pi bit for
    bit, and D3 >= 0.

log mu (and, for the reference route, the row's log-sum-exp) comes from
torch's bf16 matmul + log_softmax with the lagged weights (the behaviour
policy of the workload), never from this library.
"""

import numpy as np
import pytest
import torch

import oracle
from invariant_logprobs_gb300 import synth
from helpers import TOL_GRAD_REL_L2, TOL_LOGPI, bits, f64, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _behaviour_logprob(H, W_mu, tokens, chunk=4096):
    """log mu of each row's token and the row's log-sum-exp under the lagged
    weights, from torch's bf16 matmul + log_softmax."""
    out = torch.empty(H.shape[0], dtype=torch.float32, device=H.device)
    lse = torch.empty(H.shape[0], dtype=torch.float32, device=H.device)
    for s in range(0, H.shape[0], chunk):
        e = min(H.shape[0], s + chunk)
        zz = (H[s:e] @ W_mu.t()).float()
        lse[s:e] = torch.logsumexp(zz, dim=-1)
        z = torch.log_softmax(zz, dim=-1)
        out[s:e] = z.gather(1, tokens[s:e].long()[:, None])[:, 0]
    return out, lse


@pytest.mark.parametrize("name,route", [("qwen1p5b_lag2", "plain"), ("qwen4b_lag64", "plain"),
                                        ("qwen1p5b_lag2", "ref"), ("qwen4b_lag64", "ref")])
def test_learner_full_size_sampled(rz, name, route):
    """route "ref": rz_loss_fwd_bwd_ref with the behaviour policy's
    log-sum-exp of every row as the reference (the bench's route)."""
    wl = synth.WORKLOADS[name]
    b = synth.make_batch(wl, device=DEV)
    T, d, V, B = b["T"], b["d"], b["V"], b["B"]
    logmu, lse_mu = _behaviour_logprob(b["H"], b["W_mu"], b["tokens"])
    A32 = oracle.group_advantage(f64(b["rewards"]), b["G"]).astype(np.float32)
    adv = torch.tensor(A32, device=DEV)
    err = rz.new_err_flag(DEV)
    if route == "ref":
        out = rz.rz_loss_fwd_bwd_ref(b["H"], b["W"], b["tokens"], logmu, lse_mu, b["cu"], adv,
                                     err_flag=err)
    else:
        out = rz.rz_loss_fwd_bwd(b["H"], b["W"], b["tokens"], logmu, b["cu"], adv, err_flag=err)
    loss2, d32, _ = rz.rz_is_loss(out["logprob"], logmu, b["cu"], adv)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert np.array_equal(bits(loss2), bits(out["loss"]))
    assert np.array_equal(bits(d32), bits(out["d3"]))
    assert out["d3"].item() >= 0.0

    rng = np.random.default_rng(123)
    rows = np.sort(rng.choice(T, 64, replace=False))
    rows[0] = 0
    rows[-1] = T - 1
    r_t = torch.as_tensor(rows, device=DEV)
    Hs = f64(b["H"][r_t])
    Wd = f64(b["W"])
    tok = f64(b["tokens"][r_t])
    lp_ref, lse_ref = oracle.token_logprob_rows(Hs, Wd, tok, np.arange(64))
    lp_got = f64(out["logprob"][r_t])
    assert np.max(np.abs(lp_got - lp_ref)) <= TOL_LOGPI

    # dH rows from the oracle: each sampled row becomes a one-token response
    # whose advantage is rescaled so the oracle's c = A' w / (n * 1) equals
    # the full batch's A_i w / (B T_i) (the loss is linear in A).
    cu = f64(b["cu"])
    seg = np.searchsorted(cu, rows, side="right") - 1
    Ti = cu[seg + 1] - cu[seg]
    n = rows.shape[0]
    A_rows = A32.astype(np.float64)[seg] * n / (B * Ti)
    sub = oracle.loss_fwd_bwd(Hs, Wd, tok, f64(logmu[r_t]), np.arange(n + 1), A_rows)
    assert np.max(np.abs(sub["logpi"] - lp_ref)) <= 1e-12
    assert rel_l2(f64(out["dH"][r_t]), sub["dH"]) <= TOL_GRAD_REL_L2

    # <dW, W> == <dH, H>
    lhs = float((out["dW"].double() * b["W"].double()).sum())
    rhs = float((out["dH"].double() * b["H"].double()).sum())
    assert abs(lhs - rhs) <= 2e-2 * max(abs(lhs), abs(rhs)), (lhs, rhs)
    # sum over the vocabulary of dW is ~0 (each dz row sums to zero)
    dW64 = out["dW"].double()
    colsum = dW64.sum(0)
    assert float(colsum.norm()) <= 1e-3 * float(dW64.abs().sum(0).norm())


def test_logits_variant_full_size_sampled(rz):
    wl = synth.WORKLOADS["moe30b_logits"]
    b = synth.make_logits_batch(wl, device=DEV)
    T, V, B = b["T"], b["V"], b["B"]
    rng = np.random.default_rng(321)
    rows = np.sort(rng.choice(T, 64, replace=False))
    rows[0], rows[-1] = 0, T - 1
    r_t = torch.as_tensor(rows, device=DEV)
    z_rows = f64(b["logits"][r_t])             # keep: the call overwrites logits
    logpi = torch.empty(T, dtype=torch.float32, device=DEV)
    for s0 in range(0, T, 8192):
        e = min(T, s0 + 8192)
        zz = torch.log_softmax(b["logits"][s0:e].float(), dim=-1)
        logpi[s0:e] = zz.gather(1, b["tokens"][s0:e].long()[:, None])[:, 0]
        del zz
    logmu = synth.logmu_near(logpi, synth.LOGMU_NOISE_STD, b["gen"])
    A32 = oracle.group_advantage(f64(b["rewards"]), b["G"]).astype(np.float32)
    adv = torch.tensor(A32, device=DEV)
    err = rz.new_err_flag(DEV)
    out = rz.rz_logits_loss_fwd_bwd(b["logits"], b["tokens"], logmu, b["cu"], adv, err_flag=err)
    loss2, d32, _ = rz.rz_is_loss(out["logprob"], logmu, b["cu"], adv)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert np.array_equal(bits(loss2), bits(out["loss"]))
    assert np.array_equal(bits(d32), bits(out["d3"]))
    cu = f64(b["cu"])
    seg = np.searchsorted(cu, rows, side="right") - 1
    Ti = cu[seg + 1] - cu[seg]
    n = rows.shape[0]
    A_rows = A32.astype(np.float64)[seg] * n / (B * Ti)
    ref = oracle.logits_loss_fwd_bwd(z_rows, f64(b["tokens"][r_t]), f64(logmu[r_t]),
                                     np.arange(n + 1), A_rows)
    assert np.max(np.abs(f64(out["logprob"][r_t]) - ref["logpi"])) <= TOL_LOGPI
    assert rel_l2(f64(b["logits"][r_t]), ref["dz"]) <= TOL_GRAD_REL_L2


def test_sampler_full_size(rz):
    """The fused sampler over the 4B-shaped batch (1,083,112 rows, the bench's
    launch configuration): every recorded log mu equals rz_token_logprob of
    the drawn token bit for bit; 48 sampled rows agree with the sampler
    oracle (near-ties aside) and are drawn the same when sampled alone."""
    from oracle import rz_sampler
    wl = synth.WORKLOADS["qwen4b_lag64"]
    b = synth.make_batch(wl, device=DEV)
    T, V = b["T"], b["V"]
    rid = torch.arange(T, device=DEV, dtype=torch.int64) * 7 + 11
    seed = 0x5EED_0000_0042
    tok, lmu = rz.rz_sample_logprob(b["H"], b["W_mu"], seed, row_ids=rid)
    lp, _ = rz.rz_token_logprob(b["H"], b["W_mu"], tok)
    torch.cuda.synchronize()
    assert int(tok.min()) >= 0 and int(tok.max()) < V
    assert np.array_equal(bits(lp), bits(lmu))
    rows = np.sort(np.random.default_rng(8).choice(T, 48, replace=False))
    r_t = torch.as_tensor(rows, device=DEV)
    want_tok, _, margin = rz_sampler.sample_rows(f64(b["H"][r_t]), f64(b["W_mu"]),
                                                 f64(rid[r_t]), seed)
    got = f64(tok[r_t])
    for i in np.nonzero(got != want_tok)[0]:
        assert margin[i] < 1e-4, (rows[i], got[i], want_tok[i], margin[i])
    assert (got == want_tok).mean() >= 0.95
    # the same rows alone: bitwise the same draws
    tok1, lmu1 = rz.rz_sample_logprob(b["H"][r_t].contiguous(), b["W_mu"], seed,
                                      row_ids=rid[r_t].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(tok1, tok[r_t]) and np.array_equal(bits(lmu1), bits(lmu[r_t]))
