"""Host-side plan for running the learner step data-parallel over responses.

The loss averages tokens within a response and responses within the batch
("REINFORCE Zero" project page, s.02 objective), so whole responses are the
unit of sharding: every response's tokens stay on one rank and its per-
response mean stays local.  With B the GLOBAL number of responses,

    L = sum_r L_r,   L_r = -(1/B) sum_{i on r} A_i mean_t w_t,

and rz_loss_fwd_bwd on rank r (which divides by its local B_r) returns L_r
when it is given the advantages scaled by B_r / B.  The gradients scale the
same way, so dW = sum_r dW_r and each rank's dH is final.  D3 is a token
mean: D3 = sum_r D3_r T_r / T.

Only the sums cross ranks (dW, and two scalars), which is the one exchange
step of the path; this module holds the bookkeeping, the exchange itself is
the caller's (e.g. a fixed-order all-reduce).
"""

import numpy as np


def plan(cu_seqlens, world):
    """Split responses into `world` contiguous ranges of about equal token
    counts.  Returns a list of (first_response, last_response_exclusive)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    B = cu.shape[0] - 1
    T = int(cu[-1])
    bounds = [0]
    for r in range(1, world):
        target = T * r / world
        i = int(np.searchsorted(cu, target, side="left"))
        i = max(bounds[-1], min(B, i))
        bounds.append(i)
    bounds.append(B)
    return [(bounds[r], bounds[r + 1]) for r in range(world)]


def local_batch(cu_seqlens, resp_range):
    """Token range [t0, t1) and rebased cu_seqlens of one rank's responses."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    i0, i1 = resp_range
    t0, t1 = int(cu[i0]), int(cu[i1])
    return t0, t1, cu[i0:i1 + 1] - t0


def advantage_scale(B_local, B_global):
    """Factor applied to a rank's advantages so that its local 1/B_local
    normalisation becomes the global 1/B."""
    return 0.0 if B_global == 0 else B_local / B_global


def combine_scalars(loss_locals, d3_locals, T_locals):
    """Global loss and D3 from per-rank values (fixed rank order)."""
    T = sum(T_locals)
    loss = 0.0
    d3 = 0.0
    for l, d, t in zip(loss_locals, d3_locals, T_locals):
        loss += l
        d3 += d * t
    return loss, (d3 / T if T > 0 else 0.0)
