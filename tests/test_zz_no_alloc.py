"""rz_token_logprob_noalloc: the rollout logprob for callers that cannot
allocate device memory (engine-owned memory pools, plug-in hosts, code
between captured graph segments).  It must give the same log pi as
rz_token_logprob -- it runs the same kernels on a scratch array built into
the library -- on consecutive calls that reuse that scratch with different
sizes, and must refuse problems larger than the scratch without launching.

Kept in its own file, collected last, so a failure here never hides the
other GPU tests.
"""

import numpy as np
import pytest
import torch

from helpers import TOL_LOGPI, bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(T, d, V, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    H = torch.randn(T, d, generator=g, device=DEV).to(torch.bfloat16)
    W = (torch.randn(V, d, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    tok = torch.randint(0, V, (T,), generator=g, device=DEV, dtype=torch.int32)
    return H, W, tok


@pytest.mark.parametrize("shapes", [((3000, 512, 151936), (7777, 256, 5000)),
                                    # decode-sized batches: the logits fit the
                                    # scratch up to 55 rows at V = 151936 (56:
                                    # the fused pass, against the workspace
                                    # entry point's decode path)
                                    ((1, 2560, 151936), (55, 2048, 151936), (56, 2048, 151936))])
def test_noalloc_matches_workspace_entry_point_twice(rz, shapes):
    for i, (T, d, V) in enumerate(shapes):
        H, W, tok = _case(T, d, V, 11 + i)
        want, want_lse = rz.rz_token_logprob(H, W, tok, lse_out=torch.empty(T, device=DEV))
        got = torch.full((T,), float("nan"), device=DEV)
        got_lse = torch.full((T,), float("nan"), device=DEV)
        err = rz.new_err_flag(DEV)
        rz.rz_token_logprob_noalloc(H, W, tok, got, lse_out=got_lse, err_flag=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        assert float((got - want).abs().max()) <= TOL_LOGPI
        assert float((got_lse - want_lse).abs().max()) <= TOL_LOGPI
        # same kernels, same launch shape: bitwise the same
        assert np.array_equal(bits(got), bits(want))


def test_noalloc_rejects_sizes_beyond_its_scratch(rz):
    cap = rz.noalloc_scratch_bytes()
    V, d = 151936, 64
    T = cap // 64 + 1  # at >= 8 vocab splits, 8 bytes each: far more than the scratch holds
    W = torch.zeros(V, d, dtype=torch.bfloat16, device=DEV)
    H = torch.zeros(T, d, dtype=torch.bfloat16, device=DEV)
    tok = torch.zeros(T, dtype=torch.int32, device=DEV)
    out = torch.zeros(T, device=DEV)
    with pytest.raises(rz.RzError) as e:
        rz.rz_token_logprob_noalloc(H, W, tok, out)
    assert e.value.status == rz.RZ_ERR_TOO_LARGE
    torch.cuda.synchronize()
    assert float(out.abs().max()) == 0.0  # nothing was launched


def test_noalloc_replays_in_a_captured_graph(rz):
    """The first call on the device (outside capture) looks up the scratch
    address; later calls may then be captured.  The replayed graph matches
    rz_token_logprob bit for bit, also after its inputs are rewritten."""
    T, d, V = 2000, 256, 151936
    H, W, tok = _case(T, d, V, 21)
    got = torch.empty(T, device=DEV)
    rz.rz_token_logprob_noalloc(H, W, tok, got)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            rz.rz_token_logprob_noalloc(H, W, tok, got)
    for k in range(2):
        if k:
            H2, _, tok2 = _case(T, d, V, 22)
            H.copy_(H2)
            tok.copy_(tok2)
        got.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        want, _ = rz.rz_token_logprob(H, W, tok)
        torch.cuda.synchronize()
        assert np.array_equal(bits(got), bits(want))
