"""Launch-class timing (rz_profile_begin / rz_profile_end): it changes no
result, counts the kernels each class launches, its classes add up to the
call's own CUDA-event time, and a call captured into a CUDA graph is not
recorded."""

import numpy as np
import pytest
import torch

from helpers import bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _batch(T, d, V, B, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    H = torch.randn(T, d, generator=g, device=DEV).to(torch.bfloat16)
    W = (torch.randn(V, d, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    tok = torch.randint(0, V, (T,), generator=g, device=DEV, dtype=torch.int32)
    cuts = torch.sort(torch.randperm(T - 1, generator=g, device=DEV)[:B - 1] + 1).values
    cu = torch.cat([torch.zeros(1, dtype=torch.int64, device=DEV), cuts.to(torch.int64),
                    torch.full((1,), T, dtype=torch.int64, device=DEV)])
    logmu = -12.0 + 0.1 * torch.randn(T, generator=g, device=DEV)
    rewards = torch.rand(B, generator=g, device=DEV)
    return H, W, tok, cu, logmu, rewards


def test_profiled_learner_step_counts_and_times(rz):
    T, d, V, B = 40000, 256, 151936, 16          # two backward chunks
    H, W, tok, cu, logmu, rewards = _batch(T, d, V, B, 5)

    def step():
        adv = rz.rz_group_advantage(rewards, 8)
        return rz.rz_loss_fwd_bwd(H, W, tok, logmu, cu, adv)

    plain = step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    rz.rz_profile_begin()
    e0.record()
    prof_out = step()
    e1.record()
    prof = rz.rz_profile_end()
    step_ms = e0.elapsed_time(e1)
    # the events change no result
    for k in ("loss", "d3", "logprob", "dH", "dW"):
        assert np.array_equal(bits(plain[k]) if plain[k].dtype == torch.float32 else
                              plain[k].cpu().view(torch.int16).numpy(),
                              bits(prof_out[k]) if prof_out[k].dtype == torch.float32 else
                              prof_out[k].cpu().view(torch.int16).numpy()), k
    launches = {k: v[1] for k, v in prof.items()}
    assert launches == {"logprob_gemm": 0, "keep_gemm": 2, "merge": 2, "dz": 2, "dH_gemm": 2,
                        "dW_gemm": 2, "logits_rows": 0, "small": 1 + 1 + 2}
    summed = sum(v[0] for v in prof.values())
    assert all(v[0] > 0 for k, v in prof.items() if launches[k] > 0)
    assert 0.85 * step_ms <= summed <= step_ms * 1.001 + 0.05, (summed, step_ms)


def test_profile_skips_captured_calls_and_rollout_counts(rz):
    T, d, V = 1000, 128, 5000
    H, W, tok, _, _, _ = _batch(T, d, V, 2, 7)
    ws = rz.alloc_workspace(rz.RZ_OP_TOKEN_LOGPROB, T, d, V, 0, DEV)
    out = torch.empty(T, device=DEV)
    rz.rz_token_logprob(H, W, tok, logprob_out=out, ws=ws)  # warm-up outside capture
    torch.cuda.synchronize()
    rz.rz_profile_begin()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            rz.rz_token_logprob(H, W, tok, logprob_out=out, ws=ws)
    assert all(v == (0.0, 0) for v in rz.rz_profile_end().values())
    g.replay()
    torch.cuda.synchronize()
    want, _ = rz.rz_token_logprob(H, W, tok)
    torch.cuda.synchronize()
    assert np.array_equal(bits(out), bits(want))
    # an eager rollout call: one GEMM launch per 38,912-row block and the merge
    rz.rz_profile_begin()
    rz.rz_token_logprob(H, W, tok, logprob_out=out, ws=ws)
    prof = rz.rz_profile_end()
    assert prof["logprob_gemm"][1] == 1 and prof["merge"][1] == 1
    assert sum(v[1] for v in prof.values()) == 2
