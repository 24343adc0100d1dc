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
step of the path.  Its order is fixed: every element of dW is added in rank
order 0, 1, ..., N-1, so dW is bitwise the same on every rank and from run to
run, whatever order a backend's own all-reduce would use.  fixed_order_sum
gathers all partials on every rank; fixed_order_allreduce moves 2(N-1)/N of
the tensor per rank instead of N-1 copies: each rank receives one slice of
every rank's partial (all-to-all), adds them in rank order (the caller's
`sum_parts`, on the GPU the library's rz_sum_partials kernel) and the summed
slices are all-gathered.

On the GPU each rank calls rz_loss_fwd_bwd_shard with its own responses
and the batch's response count (so its dH rows are final and bitwise the
unsharded call's); scaling the advantages by B_r / B (advantage_scale) and
calling rz_loss_fwd_bwd gives the same step up to rounding.
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


def fixed_order_sum(t, group=None):
    """Sum of tensor t over the ranks of `group`, added in rank order
    0, 1, ..., N-1 on every rank: an all-gather of the partials, then a
    serial sum.  The result is bitwise identical on every rank and from run
    to run (a backend all-reduce may add in any order).  Holds N copies of t
    while it runs."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    parts = [torch.empty_like(t) for _ in range(world)]
    dist.all_gather(parts, t.contiguous(), group=group)
    out = parts[0].clone()
    for part in parts[1:]:
        out += part
    return out


def fixed_order_allreduce(t, sum_parts, group=None):
    """Sum of tensor t over the ranks of `group`, every element added in rank
    order 0..N-1, bitwise the same on every rank as fixed_order_sum gives.

    Element range j (of N about equal ranges) is owned by rank j: an
    all-to-all hands rank j range j of every rank's partial as the rows of
    an [N, n_j] tensor, sum_parts adds the rows in row order, and an
    all-gather returns every owner's sum to every rank.  sum_parts(parts)
    -> parts[0] + parts[1] + ... (left to right) is the only arithmetic; on
    CUDA tensors pass the library's rz_sum_partials."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    flat = t.contiguous().view(-1)
    if world == 1:
        return sum_parts(flat.view(1, -1)).view_as(t)
    n = flat.numel()
    per = -(-n // world)
    per = -(-per // 4) * 4  # 16-byte rows for the sum kernel
    send = flat
    if per * world != n:
        send = torch.cat([flat, flat.new_zeros(per * world - n)])
    recv = torch.empty(world * per, dtype=flat.dtype, device=flat.device)
    dist.all_to_all_single(recv, send, group=group)
    mine = sum_parts(recv.view(world, per)).contiguous()
    out = torch.empty(world * per, dtype=flat.dtype, device=flat.device)
    dist.all_gather_into_tensor(out, mine, group=group)
    return out[:n].view_as(t)


def dp_exchange(dW, loss, d3, sum_parts, group=None):
    """The data-parallel learner's exchange step after every rank has run
    its shard (rz_loss_fwd_bwd_shard): dW summed over ranks in rank order
    (fixed_order_allreduce) and every rank's (loss share, D3) gathered.
    loss and d3 are 1-element tensors on dW's device.  Returns (dW_sum,
    gathered [N, 2]); the batch's loss is gathered[:, 0].sum() and its D3
    the token-weighted mean of gathered[:, 1] (combine_scalars)."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    dW_sum = fixed_order_allreduce(dW, sum_parts, group)
    scal = torch.cat([loss.reshape(1), d3.reshape(1)]).to(torch.float32)
    gathered = torch.empty((world, 2), dtype=torch.float32, device=scal.device)
    dist.all_gather_into_tensor(gathered.view(-1), scal, group=group)
    return dW_sum, gathered
