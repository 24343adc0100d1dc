"""Seeded synthetic inputs shaped like the REINFORCE Zero workloads.

This module only draws inputs.  It holds none of the method's arithmetic
(no log-softmax, no importance weights, no loss); where a workload asks for
tokens "sampled from the behaviour policy" it calls torch's own matmul,
softmax and multinomial sampler as black boxes to draw them.  Both the CUDA
library and the CPU oracle receive the same arrays from here.

Workloads (stand-ins for the pages' runs; no dataset or trained weight is
used):

* ``tiny``      2 prompts x group 4, lengths U{16..64}, d=256, V=1024,
                H ~ N(0,1), W ~ N(0,0.02) (bf16), uniform tokens,
                Bernoulli(0.5) rewards, W_mu = W + N(0,1e-3).
* ``qwen1p5b_lag2``  32 x 8 responses, lengths U{256..8192}, d=1536,
                V=151936, tokens sampled from softmax(H W_mu^T),
                Bernoulli(0.4) rewards, W_mu = W + 2 steps of N(0,5e-4).
* ``qwen4b_lag64``   16 x 8 responses, lengths U{1024..16384}, d=2560,
                V=151936, sampled tokens, U[0,1] rewards,
                W_mu = W + 64 steps of N(0,2e-4).
* ``invariance_d2048``  probe rows for the batch-invariance sweep: d=2048,
                V=151936, batch sizes 1, 7, 64, 513, 4096.
* ``moe30b_logits``  given bf16 logits [262144, 151936] ~ N(0,3),
                16 x 16 responses of 1024 tokens, Bernoulli(0.3) rewards,
                uniform tokens, log mu = log pi + N(0, 0.05).

N(0, s) always means standard deviation s.  A sum of k independent
N(0, s) drift steps is drawn as one N(0, s*sqrt(k)) draw (same law).
"""

from dataclasses import dataclass, replace
import math

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    n_prompts: int
    group: int
    len_lo: int
    len_hi: int
    d: int
    V: int
    reward: str          # "bernoulli" or "uniform"
    reward_p: float
    tokens: str          # "uniform" or "sample_mu"
    drift_steps: int
    drift_std: float
    seed: int
    h_std: float = 1.0
    w_std: float = 0.02

    @property
    def B(self):
        return self.n_prompts * self.group


WORKLOADS = {
    "tiny": Workload("tiny", 2, 4, 16, 64, 256, 1024, "bernoulli", 0.5,
                     "uniform", 1, 1e-3, 1001),
    "qwen1p5b_lag2": Workload("qwen1p5b_lag2", 32, 8, 256, 8192, 1536, 151936,
                              "bernoulli", 0.4, "sample_mu", 2, 5e-4, 1002),
    "qwen4b_lag64": Workload("qwen4b_lag64", 16, 8, 1024, 16384, 2560, 151936,
                             "uniform", 0.0, "sample_mu", 64, 2e-4, 1003),
    "invariance_d2048": Workload("invariance_d2048", 1, 1, 1, 1, 2048, 151936,
                                 "bernoulli", 0.5, "uniform", 0, 0.0, 1004),
    "moe30b_logits": Workload("moe30b_logits", 16, 16, 1024, 1024, 0, 151936,
                              "bernoulli", 0.3, "uniform", 0, 0.0, 1005),
}

INVARIANCE_BATCH_SIZES = (1, 7, 64, 513, 4096)
INVARIANCE_PROBES = 64
LOGITS_STD = 3.0
LOGMU_NOISE_STD = 0.05


def scaled(wl, n_prompts=None, len_lo=None, len_hi=None, d=None, V=None,
           seed=None):
    """A smaller copy of a workload for checks the CPU oracle finishes
    quickly (same distributions, fewer/shorter responses or smaller d, V)."""
    kw = {}
    for k, v in (("n_prompts", n_prompts), ("len_lo", len_lo),
                 ("len_hi", len_hi), ("d", d), ("V", V), ("seed", seed)):
        if v is not None:
            kw[k] = v
    return replace(wl, **kw)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn_bf16(shape, std, g, device, chunk_rows=1 << 16):
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    rows = shape[0]
    for s in range(0, rows, chunk_rows):
        e = min(rows, s + chunk_rows)
        x = torch.randn((e - s,) + tuple(shape[1:]), generator=g,
                        device=device, dtype=torch.float32)
        out[s:e] = (x * std).to(torch.bfloat16)
    return out


def response_lengths(wl, g, device="cpu"):
    """T_i ~ U{len_lo .. len_hi} (inclusive), one per response."""
    return torch.randint(wl.len_lo, wl.len_hi + 1, (wl.B,), generator=g,
                         device=device, dtype=torch.int64)


def cu_from_lengths(lengths):
    cu = torch.zeros(lengths.shape[0] + 1, dtype=torch.int64,
                     device=lengths.device)
    cu[1:] = torch.cumsum(lengths, 0)
    return cu


def rewards_for(wl, g, device="cpu"):
    if wl.reward == "bernoulli":
        u = torch.rand(wl.B, generator=g, device=device)
        return (u < wl.reward_p).to(torch.float32)
    return torch.rand(wl.B, generator=g, device=device, dtype=torch.float32)


def sample_tokens_from(H, W_mu, g, chunk_rows=4096):
    """Draw a_t ~ softmax(h_t W_mu^T) with torch's sampler, row chunk by row
    chunk (the behaviour policy of the workload)."""
    T = H.shape[0]
    out = torch.empty(T, dtype=torch.int32, device=H.device)
    Wt = W_mu.t()
    for s in range(0, T, chunk_rows):
        e = min(T, s + chunk_rows)
        if H.device.type == "cuda":
            z = (H[s:e] @ Wt).float()
        else:
            z = H[s:e].float() @ Wt.float()
        probs = torch.softmax(z, dim=-1)
        out[s:e] = torch.multinomial(probs, 1, generator=g)[:, 0].to(torch.int32)
    return out


def make_batch(wl, device="cpu", seed=None, with_mu_weights=True):
    """One learner batch: H [T,d] bf16, W [V,d] bf16, W_mu [V,d] bf16,
    tokens [T] int32, cu_seqlens [B+1] int64, rewards [B] fp32."""
    g = _gen(device, wl.seed if seed is None else seed)
    lengths = response_lengths(wl, g, device)
    cu = cu_from_lengths(lengths)
    T = int(cu[-1].item())
    H = _randn_bf16((T, wl.d), wl.h_std, g, device)
    W = _randn_bf16((wl.V, wl.d), wl.w_std, g, device)
    W_mu = None
    if with_mu_weights or wl.tokens == "sample_mu":
        drift = wl.drift_std * math.sqrt(max(wl.drift_steps, 0))
        W_mu = W
        if drift > 0:
            eps = _randn_bf16((wl.V, wl.d), 1.0, g, device)
            W_mu = (W.float() + eps.float() * drift).to(torch.bfloat16)
    if wl.tokens == "uniform":
        tokens = torch.randint(0, wl.V, (T,), generator=g, device=device,
                               dtype=torch.int32)
    else:
        tokens = sample_tokens_from(H, W_mu, g)
    rewards = rewards_for(wl, g, device)
    return {"H": H, "W": W, "W_mu": W_mu, "tokens": tokens, "cu": cu,
            "rewards": rewards, "T": T, "B": wl.B, "G": wl.group,
            "d": wl.d, "V": wl.V}


def make_invariance_probes(d, V, n_probes=INVARIANCE_PROBES, device="cpu",
                           seed=1004, w_std=0.02):
    """Probe rows and weights for the batch-invariance sweep."""
    g = _gen(device, seed)
    H = _randn_bf16((n_probes, d), 1.0, g, device)
    W = _randn_bf16((V, d), w_std, g, device)
    tokens = torch.randint(0, V, (n_probes,), generator=g, device=device,
                           dtype=torch.int32)
    return H, W, tokens


def make_invariance_batch(probe_H, probe_tok, batch, g, device="cpu"):
    """Embed a random subset of probe rows at random positions among random
    co-rows; returns (H, tokens, positions, probe_index)."""
    d = probe_H.shape[1]
    n = probe_H.shape[0]
    k = min(n, batch)
    probe_idx = torch.randperm(n, generator=g, device=device)[:k]
    pos = torch.randperm(batch, generator=g, device=device)[:k]
    H = _randn_bf16((batch, d), 1.0, g, device)
    V_hi = int(probe_tok.max().item()) + 1
    tokens = torch.randint(0, max(V_hi, 1), (batch,), generator=g,
                           device=device, dtype=torch.int32)
    H[pos] = probe_H[probe_idx]
    tokens[pos] = probe_tok[probe_idx]
    return H, tokens, pos, probe_idx


def make_logits_batch(wl, device="cpu", seed=None, T=None, chunk_rows=8192):
    """Given-logits workload: logits [T,V] bf16 ~ N(0, 3), uniform tokens,
    cu_seqlens of equal 1024-token responses, rewards.  log mu is drawn by
    logmu_near() once log pi is known to the caller's harness."""
    g = _gen(device, wl.seed if seed is None else seed)
    if T is None:
        T = wl.B * wl.len_lo
    B = max(1, T // wl.len_lo) if T >= wl.len_lo else 1
    lengths = torch.full((B,), T // B, dtype=torch.int64, device=device)
    lengths[-1] += T - int(lengths.sum().item())
    cu = cu_from_lengths(lengths)
    logits = _randn_bf16((T, wl.V), LOGITS_STD, g, device, chunk_rows)
    tokens = torch.randint(0, wl.V, (T,), generator=g, device=device,
                           dtype=torch.int32)
    wl_b = replace(wl, n_prompts=max(1, B // wl.group) if B % wl.group == 0 else B,
                   group=wl.group if B % wl.group == 0 else 1)
    rewards = rewards_for(wl_b, g, device)
    return {"logits": logits, "tokens": tokens, "cu": cu, "rewards": rewards,
            "T": T, "B": B, "G": wl_b.group, "V": wl.V, "gen": g}


def logmu_near(logpi, std, g):
    """log mu = log pi + N(0, std) (the given-logits workload's behaviour
    logprobs: a recorded log mu close to the learner's)."""
    noise = torch.randn(logpi.shape, generator=g, device=logpi.device,
                        dtype=torch.float32)
    return (logpi.float() + noise * std).to(torch.float32)
