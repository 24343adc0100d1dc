"""The rollout and learner entry points inside a captured CUDA graph: they
allocate nothing and never synchronise the host, so a graph captured once
replays them exactly -- bit for bit the eager results, also after the
inputs are rewritten in place between replays."""

import numpy as np
import pytest
import torch

from helpers import bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(g, T, d, V):
    H = torch.randn(T, d, generator=g, device=DEV).to(torch.bfloat16)
    W = (torch.randn(V, d, generator=g, device=DEV) * 0.05).to(torch.bfloat16)
    tok = torch.randint(0, V, (T,), generator=g, device=DEV, dtype=torch.int32)
    return H, W, tok


@pytest.mark.parametrize("route", ["plain", "ref"])
def test_rollout_and_learner_replay_bitwise(rz, route):
    T, d, V, B = 1500, 256, 5003, 6
    g = torch.Generator(device=DEV)
    g.manual_seed(31)
    H, W, tok = _inputs(g, T, d, V)
    cu = torch.tensor([0, 100, 400, 401, 900, 1200, 1500], dtype=torch.int64, device=DEV)
    adv = torch.randn(B, generator=g, device=DEV)
    logmu = torch.empty(T, device=DEV)
    lse = torch.empty(T, device=DEV)  # the rollout's log-sum-exp (the reference route's input)

    # buffers the graph will own
    ws_r = rz.alloc_workspace(rz.RZ_OP_TOKEN_LOGPROB, T, d, V, 0, DEV)
    op = rz.RZ_OP_LOSS_FWD_BWD_REF if route == "ref" else rz.RZ_OP_LOSS_FWD_BWD
    ws_l = rz.alloc_workspace(op, T, d, V, B, DEV)
    lp = torch.empty(T, device=DEV)
    dH = torch.empty(T, d, dtype=torch.bfloat16, device=DEV)
    dW = torch.empty(V, d, device=DEV)
    loss = torch.empty(1, device=DEV)
    d3 = torch.empty(1, device=DEV)

    def work():
        rz.rz_token_logprob(H, W, tok, logprob_out=logmu, lse_out=lse, ws=ws_r)
        logmu.add_(-0.01)  # a small recorded-vs-learner gap, inside the graph too
        if route == "ref":
            rz.rz_loss_fwd_bwd_ref(H, W, tok, logmu, lse, cu, adv, logprob_out=lp, dH=dH, dW=dW,
                                   loss_out=loss, d3_out=d3, ws=ws_l)
        else:
            rz.rz_loss_fwd_bwd(H, W, tok, logmu, cu, adv, logprob_out=lp, dH=dH, dW=dW,
                               loss_out=loss, d3_out=d3, ws=ws_l)

    def snapshot():
        torch.cuda.synchronize()
        return [x.clone() for x in (logmu, lp, dH, dW, loss, d3)]

    work()
    eager = snapshot()

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        work()  # warm-up on the side stream, as graph capture expects
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        work()
    for x in (logmu, lp, dH, dW, loss, d3):
        x.zero_()
    graph.replay()
    replay = snapshot()
    for a, b in zip(eager, replay):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))

    # new inputs written in place, then replay vs eager on the same inputs
    H.copy_(torch.randn(T, d, generator=g, device=DEV).to(torch.bfloat16))
    tok.copy_(torch.randint(0, V, (T,), generator=g, device=DEV, dtype=torch.int32))
    graph.replay()
    replay2 = snapshot()
    work()
    eager2 = snapshot()
    for a, b in zip(eager2, replay2):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert not np.array_equal(bits(replay2[1]), bits(replay[1]))  # the inputs did change


@pytest.mark.parametrize("T", [1, 64])
def test_decode_sized_calls_replay_bitwise(rz, T):
    """Decode-sized rollout and sampling calls (at most 64 rows: logits GEMM,
    then the fold-and-merge kernel, each launched to overlap the kernel ahead
    of it) captured back to back in one graph: the replay matches the eager
    calls bit for bit, also after the inputs are rewritten in place."""
    d, V, steps = 256, 151936, 3
    g = torch.Generator(device=DEV)
    g.manual_seed(77 + T)
    H, W, tok = _inputs(g, T, d, V)
    rid = torch.arange(T, device=DEV, dtype=torch.int64) * 7 + 3
    ws_r = rz.alloc_workspace(rz.RZ_OP_TOKEN_LOGPROB, T, d, V, 0, DEV)
    ws_s = rz.alloc_workspace(rz.RZ_OP_SAMPLE, T, d, V, 0, DEV)
    lps = [torch.empty(T, device=DEV) for _ in range(steps)]
    lses = [torch.empty(T, device=DEV) for _ in range(steps)]
    toks = [torch.empty(T, dtype=torch.int32, device=DEV) for _ in range(steps)]
    lmus = [torch.empty(T, device=DEV) for _ in range(steps)]

    def work():
        for k in range(steps):
            rz.rz_sample_logprob(H, W, 11 + k, row_ids=rid, tokens_out=toks[k],
                                 logprob_out=lmus[k], ws=ws_s)
            rz.rz_token_logprob(H, W, tok, logprob_out=lps[k], lse_out=lses[k], ws=ws_r)

    def snapshot():
        torch.cuda.synchronize()
        return [x.clone() for x in lps + lses + toks + lmus]

    work()
    eager = snapshot()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        work()
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        work()
    for x in lps + lses + lmus:
        x.fill_(float("nan"))
    graph.replay()
    replay = snapshot()
    for a, b in zip(eager, replay):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    # each sampled token's recorded log mu is the rollout's log pi of it
    lp_s, _ = rz.rz_token_logprob(H, W, toks[0])
    torch.cuda.synchronize()
    assert np.array_equal(bits(lp_s), bits(lmus[0]))

    H.copy_(torch.randn(T, d, generator=g, device=DEV).to(torch.bfloat16))
    tok.copy_(torch.randint(0, V, (T,), generator=g, device=DEV, dtype=torch.int32))
    graph.replay()
    replay2 = snapshot()
    work()
    eager2 = snapshot()
    for a, b in zip(eager2, replay2):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
