"""Data-parallel sharding of the learner step over responses, checked on CPU
with two gloo ranks: each rank runs the oracle on its own responses with
advantages rescaled to the global batch, the ranks sum dW and the two
scalars, and the result must equal the unsharded step."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from invariant_logprobs_gb300 import shard


def _problem(seed=3):
    rng = np.random.default_rng(seed)
    B, d, V = 10, 6, 17
    L = rng.integers(0, 9, B)
    cu = np.concatenate([[0], np.cumsum(L)]).astype(np.int64)
    T = int(cu[-1])
    H = rng.standard_normal((T, d))
    W = rng.standard_normal((V, d)) * 0.5
    tok = rng.integers(0, V, T)
    lm = oracle.token_logprob(H, W + rng.standard_normal((V, d)) * 0.1, tok)[0]
    A = oracle.group_advantage(rng.random(B), 5)
    return H, W, tok, lm, cu, A


def test_plan_covers_all_responses_in_order():
    cu = np.array([0, 5, 5, 9, 30, 31, 40])
    for world in (1, 2, 3, 4, 8):
        p = shard.plan(cu, world)
        assert p[0][0] == 0 and p[-1][1] == 6
        assert all(p[i][1] == p[i + 1][0] for i in range(world - 1))
        assert all(a <= b for a, b in p)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    H, W, tok, lm, cu, A = _problem()
    B = A.shape[0]
    r0, r1 = shard.plan(cu, world)[rank]
    t0, t1, cu_l = shard.local_batch(cu, (r0, r1))
    Bl = r1 - r0
    A_l = A[r0:r1] * shard.advantage_scale(Bl, B)
    if Bl > 0:
        res = oracle.loss_fwd_bwd(H[t0:t1], W, tok[t0:t1], lm[t0:t1], cu_l, A_l)
        loss, d3, dW = res["loss"], res["d3"], res["dW"]
        dH = res["dH"]
    else:
        loss, d3, dW, dH = 0.0, 0.0, np.zeros_like(W), np.zeros((0, W.shape[1]))
    dW_t = shard.fixed_order_sum(torch.tensor(dW))
    scal = [None] * world
    dist.all_gather_object(scal, (loss, d3, t1 - t0))
    g_loss, g_d3 = shard.combine_scalars([s[0] for s in scal], [s[1] for s in scal],
                                         [s[2] for s in scal])
    np.save(os.path.join(out_dir, "dH_%d.npy" % rank), dH)
    if rank == 0:
        np.save(os.path.join(out_dir, "dW.npy"), dW_t.numpy())
        np.save(os.path.join(out_dir, "scalars.npy"), np.array([g_loss, g_d3]))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_two_rank_gloo_shard_equals_unsharded(tmp_path, world):
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    H, W, tok, lm, cu, A = _problem()
    ref = oracle.loss_fwd_bwd(H, W, tok, lm, cu, A)
    g_loss, g_d3 = np.load(tmp_path / "scalars.npy")
    assert g_loss == pytest.approx(ref["loss"], abs=1e-13)
    assert g_d3 == pytest.approx(ref["d3"], abs=1e-13)
    np.testing.assert_allclose(np.load(tmp_path / "dW.npy"), ref["dW"], atol=1e-13)
    dH = np.concatenate([np.load(tmp_path / ("dH_%d.npy" % r)) for r in range(world)])
    np.testing.assert_allclose(dH, ref["dH"], atol=1e-13)


def _partial(rank, n=4096):
    """A rank's fp32 partial whose sum depends on the order of addition
    (magnitudes from 1e-4 to 1e4)."""
    g = torch.Generator().manual_seed(100 + rank)
    return torch.randn(n, generator=g) * torch.pow(10.0, torch.randint(-4, 5, (n,), generator=g))


def _serial_sum(parts):
    """parts[0] + parts[1] + ... in row order (the exchange's rank-order sum,
    on the host for these CPU ranks)."""
    out = parts[0].clone()
    for r in range(1, parts.shape[0]):
        out += parts[r]
    return out


def _sum_worker(rank, world, port, out_dir, n=4096):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    out = shard.fixed_order_sum(_partial(rank, n))
    np.save(os.path.join(out_dir, "sum_%d.npy" % rank), out.numpy())
    # the bandwidth-optimal exchange: the same bits (a 2-D tensor whose size
    # does not divide by the rank count, so the last owner's range is ragged)
    t = _partial(rank, n).view(-1, 8)[:-1]
    out2 = shard.fixed_order_allreduce(t, _serial_sum)
    np.save(os.path.join(out_dir, "ar_%d.npy" % rank), out2.numpy())
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_fixed_order_sum_is_the_rank_order_sum_on_every_rank(tmp_path, world):
    mp.spawn(_sum_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    want = _partial(0).clone()
    for r in range(1, world):
        want += _partial(r)
    # a different order gives different bits, so the check can fail
    rev = _partial(world - 1).clone()
    for r in range(world - 2, -1, -1):
        rev += _partial(r)
    if world > 2:
        assert not torch.equal(rev, want)
    want2 = want.view(-1, 8)[:-1]
    for r in range(world):
        got = torch.from_numpy(np.load(tmp_path / ("sum_%d.npy" % r)))
        assert torch.equal(got.view(torch.int32), want.view(torch.int32)), r
        got2 = torch.from_numpy(np.load(tmp_path / ("ar_%d.npy" % r)))
        assert got2.shape == want2.shape
        assert torch.equal(got2.view(torch.int32), want2.view(torch.int32)), r


def _exchange_worker(rank, world, port, out_dir):
    """Each rank: the oracle on its shard with the global normalisation
    (advantages scaled by B_r/B), then the bench's exchange step."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    H, W, tok, lm, cu, A = _problem(5)
    B = A.shape[0]
    r0, r1 = shard.plan(cu, world)[rank]
    t0, t1, cu_l = shard.local_batch(cu, (r0, r1))
    A_l = A[r0:r1] * shard.advantage_scale(r1 - r0, B)
    res = oracle.loss_fwd_bwd(H[t0:t1], W, tok[t0:t1], lm[t0:t1], cu_l, A_l)
    dW = torch.tensor(res["dW"], dtype=torch.float32)
    dW_sum, gathered = shard.dp_exchange(dW, torch.tensor([res["loss"]]),
                                         torch.tensor([res["d3"]]), _serial_sum)
    T_r = [None] * world
    dist.all_gather_object(T_r, t1 - t0)
    loss, d3 = shard.combine_scalars(gathered[:, 0].double().tolist(),
                                     gathered[:, 1].double().tolist(), T_r)
    np.save(os.path.join(out_dir, "ex_dW_%d.npy" % rank), dW_sum.numpy())
    np.save(os.path.join(out_dir, "ex_sc_%d.npy" % rank), np.array([loss, d3]))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_dp_exchange_of_sharded_steps(tmp_path, world):
    """The bench's exchange on gloo ranks: every rank ends with the same dW
    bits, equal to the rank-order sum of the partials, and the batch's loss
    and D3 match the unsharded oracle."""
    mp.spawn(_exchange_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
             join=True)
    H, W, tok, lm, cu, A = _problem(5)
    ref = oracle.loss_fwd_bwd(H, W, tok, lm, cu, A)
    dWs = [np.load(tmp_path / ("ex_dW_%d.npy" % r)) for r in range(world)]
    for r in range(1, world):
        assert np.array_equal(dWs[r].view(np.int32), dWs[0].view(np.int32))
    np.testing.assert_allclose(dWs[0], ref["dW"], rtol=1e-5, atol=1e-6)
    for r in range(world):
        loss, d3 = np.load(tmp_path / ("ex_sc_%d.npy" % r))
        assert loss == pytest.approx(ref["loss"], rel=1e-6, abs=1e-8)
        assert d3 == pytest.approx(ref["d3"], rel=1e-6, abs=1e-8)
