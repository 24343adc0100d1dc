"""The seeded synthetic inputs follow the stated recipe (shapes, lengths,
groups, drift scale, sampling law, noise scale) and are reproducible: the
benchmark's stand-ins for the pages' workloads are what they claim to be.
CPU only, small scaled copies of the workloads."""

import math
from dataclasses import replace

import torch

from invariant_logprobs_gb300 import synth


def test_workload_table_matches_the_recipe():
    w = synth.WORKLOADS
    c2, c3, c5 = w["qwen1p5b_lag2"], w["qwen4b_lag64"], w["moe30b_logits"]
    assert (c2.B, c2.group, c2.len_lo, c2.len_hi, c2.d, c2.V) == (256, 8, 256, 8192, 1536, 151936)
    assert (c2.drift_steps, c2.drift_std, c2.tokens, c2.reward_p) == (2, 5e-4, "sample_mu", 0.4)
    assert (c3.B, c3.group, c3.len_lo, c3.len_hi, c3.d, c3.V) == (128, 8, 1024, 16384, 2560, 151936)
    assert (c3.drift_steps, c3.drift_std, c3.tokens, c3.reward) == (64, 2e-4, "sample_mu", "uniform")
    assert (c5.B, c5.group, c5.len_lo, c5.V) == (256, 16, 1024, 151936)
    assert synth.INVARIANCE_BATCH_SIZES == (1, 7, 64, 513, 4096)


def _small(name, **kw):
    base = dict(n_prompts=3, len_lo=5, len_hi=40, d=64, V=512)
    base.update(kw)
    return synth.scaled(synth.WORKLOADS[name], **base)


def test_batch_structure_and_reproducibility():
    wl = _small("qwen4b_lag64")
    a = synth.make_batch(wl)
    b = synth.make_batch(wl)
    for k in ("H", "W", "W_mu", "tokens", "cu", "rewards"):
        assert torch.equal(a[k], b[k]), k
    c = synth.make_batch(wl, seed=wl.seed + 1)
    assert not torch.equal(a["H"], c["H"])
    cu, T = a["cu"], a["T"]
    lengths = cu[1:] - cu[:-1]
    assert cu[0] == 0 and cu[-1] == T and len(cu) == wl.B + 1
    assert int(lengths.min()) >= wl.len_lo and int(lengths.max()) <= wl.len_hi
    assert a["H"].shape == (T, wl.d) and a["H"].dtype == torch.bfloat16
    assert a["W"].shape == (wl.V, wl.d) and a["W_mu"].shape == (wl.V, wl.d)
    assert int(a["tokens"].min()) >= 0 and int(a["tokens"].max()) < wl.V
    assert a["tokens"].dtype == torch.int32 and a["rewards"].shape == (wl.B,)
    assert float(a["rewards"].min()) >= 0.0 and float(a["rewards"].max()) <= 1.0
    assert a["G"] == wl.group and wl.B % wl.group == 0


def test_behaviour_weights_drift_by_sigma_sqrt_steps():
    for name in ("qwen1p5b_lag2", "qwen4b_lag64"):
        wl = _small(name, d=128, V=1024)
        b = synth.make_batch(wl)
        diff = b["W_mu"].float() - b["W"].float()
        want = wl.drift_std * math.sqrt(wl.drift_steps)
        # bf16 rounding of W_mu adds ~2^-9 |W| of noise: compare with it removed
        rounding = 2.0 ** -9 * b["W"].float().abs().mean().item()
        got = diff.std().item()
        assert abs(got - want) <= 0.1 * want + rounding, (name, got, want)
    tiny = synth.make_batch(synth.WORKLOADS["tiny"])
    assert tiny["W_mu"] is not None


def test_sampled_tokens_follow_the_behaviour_softmax():
    # large enough weights that softmax(H W_mu^T) is far from uniform
    wl = replace(_small("qwen4b_lag64", n_prompts=4, len_lo=200, len_hi=200, d=32, V=64),
                 w_std=0.5)
    b = synth.make_batch(wl)
    z = b["H"].float() @ b["W_mu"].float().t()
    p = torch.softmax(z, dim=-1)
    picked = p.gather(1, b["tokens"].long()[:, None])[:, 0]
    # E[p(a)] under a ~ p is sum p^2; under uniform tokens it would be 1/V
    expect = (p * p).sum(1).mean().item()
    assert abs(picked.mean().item() - expect) < 0.15 * expect
    assert picked.mean().item() > 4.0 / wl.V


def test_invariance_batch_places_the_probes():
    H, W, tok = synth.make_invariance_probes(32, 300, n_probes=16)
    g = torch.Generator().manual_seed(5)
    for batch in (1, 7, 64):
        Hb, tb, pos, idx = synth.make_invariance_batch(H, tok, batch, g)
        assert Hb.shape == (batch, 32) and tb.shape == (batch,)
        assert len(set(pos.tolist())) == len(pos) == min(16, batch)
        assert torch.equal(Hb[pos], H[idx]) and torch.equal(tb[pos], tok[idx])
        assert int(tb.max()) < 300


def test_logits_batch_and_logmu_noise():
    wl = synth.WORKLOADS["moe30b_logits"]
    b = synth.make_logits_batch(replace(wl, V=4096), T=4096)
    assert b["logits"].shape == (4096, 4096) and b["cu"][-1] == 4096
    lengths = b["cu"][1:] - b["cu"][:-1]
    assert int(lengths.min()) == int(lengths.max()) == wl.len_lo
    assert abs(b["logits"].float().std().item() - synth.LOGITS_STD) < 0.05
    assert b["rewards"].shape == (b["B"],) and b["B"] % b["G"] == 0
    lp = torch.zeros(100000)
    lm = synth.logmu_near(lp, synth.LOGMU_NOISE_STD, torch.Generator().manual_seed(1))
    assert abs(lm.std().item() - synth.LOGMU_NOISE_STD) < 0.002
    assert abs(lm.mean().item()) < 0.002
