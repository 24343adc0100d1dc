"""Decode-sized batches (at most 64 rows).  Given a workspace with room for
the batch's fp32 logits, rz_token_logprob and rz_sample_logprob compute the
logits with one vocabulary tile per task and then fold and merge them in a
second kernel (one cluster of CTAs per row, one warp per vocabulary split).
The vocabularies below give one split (a single tile, a ragged one), a few
splits, all 64 splits of one tile each, and splits of several tiles with a
ragged last tile; the results must be the fused pass's bit for bit (the same
call on a workspace without that room) and match the oracle."""

import numpy as np
import pytest
import torch

import oracle
from helpers import TOL_LOGPI, bits, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"

# V -> vocabulary splits (tiles of 256 columns, at most 64 splits):
# 8 -> 1, 256 -> 1, 1000 -> 4, 16384 -> 64, 20000 -> 40 (2 tiles each),
# 151936 -> 60 (10 tiles each, the last split 4)
VOCABS = [8, 256, 1000, 16384, 20000, 151936]


def _inputs(T, d, V, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    H = torch.randn(T, d, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, d, generator=g) * (scale / np.sqrt(d))).to(torch.bfloat16)
    tok = torch.randint(0, V, (T,), generator=g, dtype=torch.int32)
    tok[0] = V - 1  # the last column, inside the ragged tail
    if T > 1:
        tok[1] = 0
    return H.to(DEV), W.to(DEV), tok.to(DEV)


def _fused_ws(rz, d, V):
    # sized for 65 rows: no room for a decode-sized batch's logits, so the
    # call keeps the fused pass
    return rz.alloc_workspace(rz.RZ_OP_TOKEN_LOGPROB, 65, d, V, 0, DEV)


@pytest.mark.parametrize("V", VOCABS)
@pytest.mark.parametrize("T", [1, 7, 64])
def test_decode_logprob_equals_fused_pass_and_oracle(rz, T, V):
    d = 128
    H, W, tok = _inputs(T, d, V, seed=T * 1000 + V)
    lp, lse = rz.rz_token_logprob(H, W, tok)  # workspace sized for T: decode mode
    lp2, lse2 = rz.rz_token_logprob(H, W, tok, ws=_fused_ws(rz, d, V))
    torch.cuda.synchronize()
    assert np.array_equal(bits(lp), bits(lp2))
    assert np.array_equal(bits(lse), bits(lse2))
    want_lp, want_lse = oracle.token_logprob(f64(H), f64(W), f64(tok))
    assert np.max(np.abs(f64(lp) - want_lp)) <= TOL_LOGPI
    assert np.max(np.abs(f64(lse) - want_lse)) <= TOL_LOGPI


@pytest.mark.parametrize("V", [1000, 151936])
def test_decode_logprob_peaked_rows(rz, V):
    # logits with a spread of ~30: log pi of the likeliest tokens near 0
    T, d = 16, 256
    H, W, _ = _inputs(T, d, V, seed=7, scale=30.0)
    z = (H.float() @ W.float().T)
    tok = z.argmax(dim=1).to(torch.int32)
    lp, _ = rz.rz_token_logprob(H, W, tok)
    lp2, _ = rz.rz_token_logprob(H, W, tok, ws=_fused_ws(rz, d, V))
    torch.cuda.synchronize()
    assert np.array_equal(bits(lp), bits(lp2))
    want, _ = oracle.token_logprob(f64(H), f64(W), f64(tok))
    assert np.max(np.abs(f64(lp) - want)) <= TOL_LOGPI
    assert float(lp.max()) > -1e-3  # some rows are peaked


@pytest.mark.parametrize("V", VOCABS)
def test_decode_sampler_equals_fused_pass(rz, V):
    T, d = 33, 128
    H, W, _ = _inputs(T, d, V, seed=V + 5)
    rid = torch.arange(T, device=DEV, dtype=torch.int64) * 104729 + 11
    tok, lmu = rz.rz_sample_logprob(H, W, 1234, row_ids=rid)  # decode mode
    ws = rz.alloc_workspace(rz.RZ_OP_SAMPLE, 65, d, V, 0, DEV)
    tok2, lmu2 = rz.rz_sample_logprob(H, W, 1234, row_ids=rid, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(tok, tok2)
    assert np.array_equal(bits(lmu), bits(lmu2))
    t = tok.cpu().numpy()
    assert t.min() >= 0 and t.max() < V
    # the recorded log mu is the rollout's log pi of the drawn token
    lp, _ = rz.rz_token_logprob(H, W, tok)
    torch.cuda.synchronize()
    assert np.array_equal(bits(lp), bits(lmu))


def test_decode_out_of_range_tokens(rz):
    T, d, V = 9, 64, 20000
    H, W, tok = _inputs(T, d, V, seed=3)
    tok[2] = V
    tok[5] = -7
    for ws in (None, _fused_ws(rz, d, V)):
        err = rz.new_err_flag(DEV)
        lp, lse = rz.rz_token_logprob(H, W, tok, ws=ws, err_flag=err)
        torch.cuda.synchronize()
        assert err.item() & rz.RZ_DEVERR_TOKEN_RANGE
        assert torch.isnan(lp[2]) and torch.isnan(lp[5])
        assert torch.isnan(lse[2]) and torch.isnan(lse[5])
        ok = [i for i in range(T) if i not in (2, 5)]
        assert bool(torch.all(torch.isfinite(lp[ok])))
