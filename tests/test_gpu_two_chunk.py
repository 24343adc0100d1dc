"""Learner parity past one backward chunk, at the full vocabulary.

The learner runs its backward pass in chunks of rows (38,912 at
V = 151936; fewer at very large vocabularies, where the chunk's kept terms
would pass 40 GiB), while the rollout's logprob GEMM runs in launch blocks
of 38,912 rows whatever V is.  These tests cross those boundaries:

  * V = 151936, d = 1536, ~43,000 rows (two chunks, the second ragged): log pi,
    the loss, D3, and dH and dW element by element against the fp64 oracle,
    as whole tensors (relative L2) and row by row (every dH row, every dW
    vocabulary row);
  * V = 151936, more than two chunks of rows: the learner's log pi equals
    the rollout's bit for bit at the same weights, so w == 1 and D3 == 0.0
    exactly ("diff 0", the Zero Mismatch post s.5);
  * a vocabulary large enough that the learner's chunk is capped below the
    rollout's launch block, so their boundaries fall on different rows: the
    same bitwise equality.

log mu for the parity case comes from torch's bf16 matmul + log_softmax
under the lagged weights (the behaviour policy of the workload), never from
this library; the advantages are the oracle's, rounded to fp32.
"""

import numpy as np
import pytest
import torch

import oracle
from invariant_logprobs_gb300 import synth
from helpers import (TOL_GRAD_REL_L2, TOL_LOGPI, bits, f64, rel_l2, scalar_close)

pytestmark = pytest.mark.gpu
DEV = "cuda"
CHUNK_ROWS = 38912          # learner chunk and rollout launch block at V = 151936
ROW_REL_L2 = 2e-2           # per dH row and per dW vocabulary row (see row_errors)


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


def row_errors(got, want):
    """Relative L2 error of every row, with a floor of 1e-3 of the root mean
    square row norm (a row whose reference is ~0 is judged on absolute
    error).  bf16 outputs and a bf16 dz give ~2-4e-3 per row; 2e-2 leaves
    room for the worst of ~150,000 rows."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    num = np.linalg.norm(got - want, axis=1)
    den = np.linalg.norm(want, axis=1)
    floor = 1e-3 * np.sqrt(np.mean(den ** 2))
    return num / np.maximum(den, floor)


def test_two_chunk_full_vocab_gradients_vs_oracle(rz):
    wl = synth.scaled(synth.WORKLOADS["qwen1p5b_lag2"], n_prompts=2, len_lo=2600,
                      len_hi=2800, seed=2203)
    b = synth.make_batch(wl, device=DEV)
    T, d, V, B = b["T"], b["d"], b["V"], b["B"]
    assert (d, V) == (1536, 151936)
    assert CHUNK_ROWS < T < 2 * CHUNK_ROWS and (T - CHUNK_ROWS) % 128 != 0
    logmu, lse_mu = _behaviour_logprob(b["H"], b["W_mu"], b["tokens"])
    A32 = oracle.group_advantage(f64(b["rewards"]), b["G"]).astype(np.float32)
    err = rz.new_err_flag(DEV)
    out = rz.rz_loss_fwd_bwd(b["H"], b["W"], b["tokens"], logmu, b["cu"],
                             torch.tensor(A32, device=DEV), err_flag=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    got = {k: f64(out[k]) for k in ("logprob", "dH", "dW")}
    loss, d3 = out["loss"].item(), out["d3"].item()
    del out
    # the same step through the per-row reference route (the behaviour
    # policy's log-sum-exp as the reference)
    out = rz.rz_loss_fwd_bwd_ref(b["H"], b["W"], b["tokens"], logmu, lse_mu, b["cu"],
                                 torch.tensor(A32, device=DEV), err_flag=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    got_ref = {k: f64(out[k]) for k in ("dH", "dW")}
    assert np.array_equal(bits(out["logprob"]), bits(torch.tensor(got["logprob"],
                                                                  dtype=torch.float32)))
    assert out["loss"].item() == loss and out["d3"].item() == d3
    del out
    torch.cuda.empty_cache()

    ref = oracle.loss_fwd_bwd(f64(b["H"]), f64(b["W"]), f64(b["tokens"]), f64(logmu),
                              f64(b["cu"]), A32.astype(np.float64))
    assert np.max(np.abs(got["logprob"] - ref["logpi"])) <= TOL_LOGPI
    assert scalar_close(loss, ref["loss"]), (loss, ref["loss"])
    assert scalar_close(d3, ref["d3"]), (d3, ref["d3"])
    e_dH, e_dW = rel_l2(got["dH"], ref["dH"]), rel_l2(got["dW"], ref["dW"])
    assert e_dH <= TOL_GRAD_REL_L2 and e_dW <= TOL_GRAD_REL_L2, (e_dH, e_dW)
    # row by row: a mis-addressed tile in either chunk, or in the ragged tail
    # of the second, shows up in its own rows even where the totals pass
    r_dH = row_errors(got["dH"], ref["dH"])
    r_dW = row_errors(got["dW"], ref["dW"])
    assert r_dH.max() <= ROW_REL_L2, (int(r_dH.argmax()), r_dH.max(), np.median(r_dH))
    assert r_dW.max() <= ROW_REL_L2, (int(r_dW.argmax()), r_dW.max(), np.median(r_dW))
    # both chunks are held to the same bar
    assert r_dH[:CHUNK_ROWS].max() <= ROW_REL_L2 and r_dH[CHUNK_ROWS:].max() <= ROW_REL_L2
    # the reference route, element by element and row by row as well
    e2_dH, e2_dW = rel_l2(got_ref["dH"], ref["dH"]), rel_l2(got_ref["dW"], ref["dW"])
    assert e2_dH <= TOL_GRAD_REL_L2 and e2_dW <= TOL_GRAD_REL_L2, (e2_dH, e2_dW)
    r2_dH = row_errors(got_ref["dH"], ref["dH"])
    r2_dW = row_errors(got_ref["dW"], ref["dW"])
    assert r2_dH.max() <= ROW_REL_L2 and r2_dW.max() <= ROW_REL_L2, (r2_dH.max(), r2_dW.max())
    print("two-chunk reference route: dH rel L2 %.2e (rows max %.2e); dW rel L2 %.2e "
          "(vocab rows max %.2e)" % (e2_dH, r2_dH.max(), e2_dW, r2_dW.max()))
    print("two-chunk T=%d: |dlogpi| max %.2e; loss rel %.2e; d3 rel %.2e; dH rel L2 %.2e "
          "(rows: median %.2e, max %.2e); dW rel L2 %.2e (vocab rows: median %.2e, max %.2e)"
          % (T, np.max(np.abs(got["logprob"] - ref["logpi"])),
             abs(loss - ref["loss"]) / abs(ref["loss"]), abs(d3 - ref["d3"]) / abs(ref["d3"]),
             e_dH, np.median(r_dH), r_dH.max(), e_dW, np.median(r_dW), r_dW.max()))


def _zero_mismatch(rz, T, d, V, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    H = (torch.randn(T, d, generator=g, device=DEV)).to(torch.bfloat16)
    W = (torch.randn(V, d, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    tokens = torch.randint(0, V, (T,), generator=g, device=DEV, dtype=torch.int32)
    n_resp = 24
    cuts = torch.sort(torch.randperm(T - 1, generator=g, device=DEV)[:n_resp - 1] + 1).values
    cu = torch.cat([torch.zeros(1, dtype=torch.int64, device=DEV), cuts.to(torch.int64),
                    torch.full((1,), T, dtype=torch.int64, device=DEV)])
    adv = rz.rz_group_advantage(torch.rand(n_resp, generator=g, device=DEV), 8)
    err = rz.new_err_flag(DEV)
    # the rollout records log mu (and each row's log-sum-exp) with the same
    # weights the learner holds
    lse = torch.empty(T, dtype=torch.float32, device=DEV)
    logmu, _ = rz.rz_token_logprob(H, W, tokens, err_flag=err, lse_out=lse)
    ws_bytes = rz.workspace_size(rz.RZ_OP_LOSS_FWD_BWD, T, d, V, n_resp)
    out = rz.rz_loss_fwd_bwd(H, W, tokens, logmu, cu, adv, err_flag=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert np.array_equal(bits(out["logprob"]), bits(logmu))
    assert out["d3"].item() == 0.0
    # the reference route over the same chunks: the same log pi, loss and D3
    # bits, gradients to rounding.  The routes round in different places
    # (bf16 terms against the reference and a scaled H, against bf16 dz), and
    # a dH element here sums up to 2^24 rounded terms before its own bf16
    # rounding; each route is held to rel L2 1e-2 against the oracle
    # (test_two_chunk_full_vocab_gradients_vs_oracle), and so is their
    # difference here (measured 5.9e-3 for dH at V = 2^24).
    out_r = rz.rz_loss_fwd_bwd_ref(H, W, tokens, logmu, lse, cu, adv, err_flag=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert np.array_equal(bits(out_r["logprob"]), bits(logmu))
    assert out_r["d3"].item() == 0.0
    assert np.array_equal(bits(out_r["loss"]), bits(out["loss"]))
    assert rel_l2(f64(out_r["dH"]), f64(out["dH"])) <= TOL_GRAD_REL_L2
    assert rel_l2(f64(out_r["dW"]), f64(out["dW"])) <= TOL_GRAD_REL_L2
    del out_r
    # w == 1 exactly: the loss is -(1/B) sum_i A_i, the same as rz_is_loss
    # gives for log pi == log mu
    loss2, d32, _ = rz.rz_is_loss(logmu, logmu, cu, adv)
    torch.cuda.synchronize()
    assert np.array_equal(bits(loss2), bits(out["loss"])) and d32.item() == 0.0
    return ws_bytes


def test_zero_mismatch_past_two_chunks_full_vocab(rz):
    T = 2 * CHUNK_ROWS + 3001
    _zero_mismatch(rz, T, 1536, 151936, 41)


def test_zero_mismatch_when_the_learner_chunk_is_capped(rz):
    # At V = 600,000 a 38,912-row chunk would keep 2.125 B x 38,912 x V > 40 GiB
    # of terms, so the learner's chunk shrinks (to 33,664 rows) while the
    # rollout still launches blocks of 38,912 rows.
    V, d = 600000, 128
    per_row = (V + 7) // 8 * 8 * 2 + (V + 127) // 128 * 4 * 4
    chunk = (40 << 30) // per_row // 128 * 128
    assert chunk < CHUNK_ROWS
    T = 2 * chunk + 5000
    ws_bytes = _zero_mismatch(rz, T, d, V, 43)
    assert ws_bytes >= chunk * per_row  # the workspace holds one capped chunk


def test_maximum_vocabulary(rz):
    """V = 2^24, the largest vocabulary the boundary accepts: the learner's
    chunk shrinks to 1,152 rows (40 GiB of kept terms), so 2,500 rows cross
    three chunks.  Rollout and learner agree bit for bit (w == 1, D3 == 0),
    sampled rows match the oracle's log pi, and the fused sampler records
    the logprob of what it draws."""
    V, d, T = 1 << 24, 16, 2500
    per_row = (V + 7) // 8 * 8 * 2 + (V + 127) // 128 * 4 * 4
    assert (40 << 30) // per_row // 128 * 128 == 1152
    ws_bytes = _zero_mismatch(rz, T, d, V, 47)
    assert ws_bytes >= 1152 * per_row
    g = torch.Generator(device=DEV).manual_seed(48)
    H = torch.randn(T, d, generator=g, device=DEV).to(torch.bfloat16)
    W = (torch.randn(V, d, generator=g, device=DEV) * 0.3).to(torch.bfloat16)
    tok = torch.randint(0, V, (T,), generator=g, device=DEV, dtype=torch.int32)
    lp, _ = rz.rz_token_logprob(H, W, tok)
    stok, slmu = rz.rz_sample_logprob(H, W, 3)
    lp_s, _ = rz.rz_token_logprob(H, W, stok)
    torch.cuda.synchronize()
    assert np.array_equal(bits(lp_s), bits(slmu))
    assert int(stok.min()) >= 0 and int(stok.max()) < V
    rows = np.array([0, 1151, 1152, T - 1])
    r_t = torch.as_tensor(rows, device=DEV)
    want, _ = oracle.token_logprob_rows(f64(H[r_t]), f64(W), f64(tok[r_t]), np.arange(4))
    assert np.max(np.abs(f64(lp[r_t]) - want)) <= TOL_LOGPI
