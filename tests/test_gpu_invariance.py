"""Bit-exact properties: batch invariance of log pi (a row's logprob is the
same float whatever batch it sits in), rollout == learner at equal weights
("diff 0": w == 1, D3 == 0), run-to-run determinism, and argument/device
error reporting."""

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from invariant_logprobs_gb300 import synth
from helpers import TOL_LOGPI, bits, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_batch_invariance_sweep(rz):
    d, V = 2048, 151936
    pH, W, ptok = synth.make_invariance_probes(d, V, device=DEV)
    g = torch.Generator(device=DEV)
    g.manual_seed(99)
    n = pH.shape[0]
    ref_bits = np.zeros(n, dtype=np.int32)
    known = np.zeros(n, dtype=bool)
    ws = rz.alloc_workspace(rz.RZ_OP_TOKEN_LOGPROB, 4096, d, V, 0, DEV)
    for batch in synth.INVARIANCE_BATCH_SIZES:
        for rep in range(2):
            H, tok, pos, pidx = synth.make_invariance_batch(pH, ptok, batch, g, DEV)
            lp, _ = rz.rz_token_logprob(H, W, tok, ws=ws)
            # a workspace sized for this batch: decode-sized batches (<= 64
            # rows) then take the logits through it and fold them apart
            lp2, _ = rz.rz_token_logprob(H, W, tok)
            torch.cuda.synchronize()
            assert np.array_equal(bits(lp), bits(lp2)), batch
            idx = pidx.cpu().numpy()
            b = bits(lp[pos])
            seen = known[idx]
            assert np.array_equal(b[seen], ref_bits[idx][seen]), (batch, rep)
            ref_bits[idx[~seen]] = b[~seen]
            known[idx] = True
    # every probe was seen (batch 4096 holds all 64) and matches the oracle
    assert np.all(known)
    lp_all, _ = rz.rz_token_logprob(pH, W, ptok)
    torch.cuda.synchronize()
    assert np.array_equal(bits(lp_all), ref_bits)
    want, _ = oracle.token_logprob(f64(pH), f64(W), f64(ptok))
    assert np.max(np.abs(f64(lp_all) - want)) <= TOL_LOGPI


def test_rollout_equals_learner_zero_mismatch(rz):
    wl = synth.scaled(synth.WORKLOADS["qwen1p5b_lag2"], n_prompts=1, len_lo=100, len_hi=700,
                      V=20000)
    wl = dataclasses.replace(wl, tokens="uniform")
    b = synth.make_batch(wl, device=DEV)
    H, W, tok, cu = b["H"], b["W"], b["tokens"], b["cu"]
    adv = rz.rz_group_advantage(b["rewards"], b["G"])
    # rollout records log mu with the SAME weights
    logmu, _ = rz.rz_token_logprob(H, W, tok)
    out = rz.rz_loss_fwd_bwd(H, W, tok, logmu, cu, adv)
    torch.cuda.synchronize()
    assert np.array_equal(bits(out["logprob"]), bits(logmu))      # diff 0
    assert out["d3"].item() == 0.0
    w = torch.exp(out["logprob"] - logmu)
    assert bool(torch.all(w == 1.0))
    # with w == 1 the loss is -mean(A) over non-empty responses
    Ti = (cu[1:] - cu[:-1]).cpu()
    A = adv.cpu()
    want = -float((A * (Ti > 0)).double().sum()) / A.shape[0]
    assert abs(out["loss"].item() - want) <= 1e-6


def test_learner_run_to_run_deterministic(rz):
    wl = synth.Workload("det", 2, 4, 300, 900, 512, 9000, "uniform", 0.0, "uniform", 4, 1e-3, 31)
    b = synth.make_batch(wl, device=DEV)
    adv = rz.rz_group_advantage(b["rewards"], b["G"])
    logmu, _ = rz.rz_token_logprob(b["H"], b["W_mu"], b["tokens"])
    outs = []
    side = torch.cuda.Stream()
    for k in range(3):
        s = side if k == 1 else torch.cuda.current_stream()
        if k == 1:
            side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            outs.append(rz.rz_loss_fwd_bwd(b["H"], b["W"], b["tokens"], logmu, b["cu"], adv))
        torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o["dH"], outs[0]["dH"])
        assert torch.equal(o["dW"], outs[0]["dW"])
        assert np.array_equal(bits(o["loss"]), bits(outs[0]["loss"]))
        assert np.array_equal(bits(o["d3"]), bits(outs[0]["d3"]))
        assert np.array_equal(bits(o["logprob"]), bits(outs[0]["logprob"]))


def test_empty_and_single_row(rz):
    d, V = 64, 512
    W = torch.randn(V, d, device=DEV).to(torch.bfloat16)
    H0 = torch.empty(0, d, dtype=torch.bfloat16, device=DEV)
    t0 = torch.empty(0, dtype=torch.int32, device=DEV)
    lp, _ = rz.rz_token_logprob(H0, W, t0)
    assert lp.numel() == 0
    cu = torch.zeros(3, dtype=torch.int64, device=DEV)
    adv = torch.tensor([0.5, -0.5], device=DEV)
    out = rz.rz_loss_fwd_bwd(H0, W, t0, torch.empty(0, device=DEV), cu, adv)
    torch.cuda.synchronize()
    assert out["loss"].item() == 0.0 and out["d3"].item() == 0.0
    assert bool(torch.all(out["dW"] == 0))
    # one row, one response
    H1 = torch.randn(1, d, device=DEV).to(torch.bfloat16)
    t1 = torch.tensor([3], dtype=torch.int32, device=DEV)
    lp1, _ = rz.rz_token_logprob(H1, W, t1)
    cu1 = torch.tensor([0, 1], dtype=torch.int64, device=DEV)
    out1 = rz.rz_loss_fwd_bwd(H1, W, t1, lp1 - 0.25, cu1, torch.tensor([2.0], device=DEV))
    torch.cuda.synchronize()
    ref = oracle.loss_fwd_bwd(f64(H1), f64(W), f64(t1), f64(lp1) - 0.25, np.array([0, 1]),
                              np.array([2.0]))
    assert abs(out1["loss"].item() - ref["loss"]) <= 1e-4 * abs(ref["loss"])


def test_device_errors_are_flagged_not_trapped(rz):
    d, V, T = 64, 300, 10
    H = torch.randn(T, d, device=DEV).to(torch.bfloat16)
    W = torch.randn(V, d, device=DEV).to(torch.bfloat16)
    tok = torch.randint(0, V, (T,), dtype=torch.int32, device=DEV)
    tok[4] = V + 5
    tok[7] = -1
    err = rz.new_err_flag(DEV)
    lp, _ = rz.rz_token_logprob(H, W, tok, err_flag=err)
    torch.cuda.synchronize()
    assert err.item() & rz.RZ_DEVERR_TOKEN_RANGE
    assert torch.isnan(lp[4]) and torch.isnan(lp[7])
    ok = [i for i in range(T) if i not in (4, 7)]
    assert bool(torch.all(torch.isfinite(lp[ok])))
    # bad cu_seqlens: decreasing
    err.zero_()
    logpi = torch.zeros(T, device=DEV)
    cu = torch.tensor([0, 6, 3, T], dtype=torch.int64, device=DEV)
    rz.rz_is_loss(logpi, logpi, cu, torch.zeros(3, device=DEV), err_flag=err)
    torch.cuda.synchronize()
    assert err.item() & rz.RZ_DEVERR_CU_SEQLENS
    # the context is still healthy
    assert torch.ones(3, device=DEV).sum().item() == 3.0


def test_host_argument_errors(rz):
    r = torch.rand(10, device=DEV)
    with pytest.raises(rz.RzError) as e:
        rz.rz_group_advantage(r, 4)
    assert e.value.status == rz.RZ_ERR_INVALID_ARG
    H = torch.randn(4, 12, device=DEV).to(torch.bfloat16)   # d % 8 != 0
    W = torch.randn(9, 12, device=DEV).to(torch.bfloat16)
    tok = torch.zeros(4, dtype=torch.int32, device=DEV)
    with pytest.raises(rz.RzError) as e:
        rz.rz_token_logprob(H, W, tok)
    assert e.value.status == rz.RZ_ERR_UNSUPPORTED
    H = torch.randn(4, 16, device=DEV).to(torch.bfloat16)
    W = torch.randn(9, 16, device=DEV).to(torch.bfloat16)
    small = torch.empty(256, dtype=torch.uint8, device=DEV)
    with pytest.raises(rz.RzError) as e:
        rz.rz_token_logprob(H, W, tok, ws=small[:1])
    assert e.value.status == rz.RZ_ERR_WORKSPACE


def test_bounded_wait_gives_up_and_reports(rz):
    """A pipeline wait on a barrier nothing completes returns after its limit
    with RZ_DEVERR_TIMEOUT set; the context remains usable."""
    import time
    err = rz.new_err_flag(DEV)
    done = torch.zeros(1, dtype=torch.int32, device=DEV)
    t0 = time.perf_counter()
    rz.rz_selftest_wait_timeout(err, done, limit_us=50000)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert err.item() & rz.RZ_DEVERR_TIMEOUT
    assert done.item() == 2
    assert 0.04 <= dt < 5.0, dt
    assert torch.arange(10, device=DEV).sum().item() == 45


def test_binding_rejects_mismatched_shapes_before_launch(rz):
    H = torch.randn(10, 16, device=DEV).to(torch.bfloat16)
    W = torch.randn(30, 16, device=DEV).to(torch.bfloat16)
    tok = torch.zeros(9, dtype=torch.int32, device=DEV)      # one short
    with pytest.raises(ValueError):
        rz.rz_token_logprob(H, W, tok)
    cu = torch.tensor([0, 4, 10], dtype=torch.int64, device=DEV)
    lm = torch.zeros(10, device=DEV)
    with pytest.raises(ValueError):
        rz.rz_loss_fwd_bwd(H, W, torch.zeros(10, dtype=torch.int32, device=DEV), lm, cu,
                           torch.zeros(3, device=DEV))             # adv has B+1 entries
    with pytest.raises(ValueError):
        rz.rz_is_loss(lm, lm[:9], cu, torch.zeros(2, device=DEV))
    W_bad = torch.randn(30, 8, device=DEV).to(torch.bfloat16)  # d mismatch
    with pytest.raises(ValueError):
        rz.rz_token_logprob(H, W_bad, torch.zeros(10, dtype=torch.int32, device=DEV))
