"""The token-sharded (data-parallel) path on CPU with two gloo ranks.

The loss shards by tokens: each rank runs the fused loss on its own tokens
with W replicated.  Per rank, the loss is the mean over that rank's valid
tokens, so the global loss and gradients come from reweighting each rank by
its share of the valid tokens and summing (dp_combine).  Here the fp64 oracle
stands in for each rank's GPU call, and the combination must reproduce the
oracle on the whole batch.  The bench's rank logic (one seed per shard, the
slowest rank's time) is checked on the same two ranks."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    import top_kl_loss_token_b300 as kd
    from top_kl_loss_token_b300 import synth
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x = synth.make_inputs(90, 32, 300, 6, T=2.0, dtype="fp32", seed=5, mask="random0.3",
                              w_std=0.3)
        # uneven shards with different valid counts
        cut = 37
        sl = slice(0, cut) if rank == 0 else slice(cut, x.N)
        m = x.mask[sl]
        r = oracle.fwd_bwd(x.h_f32()[sl], x.W_f32(), x.idx[sl], x.logit[sl], m, x.T)
        loss = torch.tensor([r["loss"]], dtype=torch.float64)
        gh = torch.from_numpy(r["grad_h"].copy())
        gW = torch.from_numpy(r["grad_W"].copy())
        kd.dp_combine(loss, gh, gW, int(m.sum()))
        # bench rank logic
        t = bench.max_over_ranks(10.0 + rank, world, "cpu")
        seeds = [bench.shard_seed(3, k, world) for k in range(world)]
        q.put((rank, float(loss.item()), gh.numpy(), gW.numpy(), t, seeds))
    finally:
        dist.destroy_process_group()


def test_token_sharded_combination_matches_whole_batch():
    import oracle
    from top_kl_loss_token_b300 import synth
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        rank, loss, gh, gW, t, seeds = q.get(timeout=120)
        res[rank] = (loss, gh, gW, t, seeds)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    x = synth.make_inputs(90, 32, 300, 6, T=2.0, dtype="fp32", seed=5, mask="random0.3",
                          w_std=0.3)
    full = oracle.fwd_bwd(x.h_f32(), x.W_f32(), x.idx, x.logit, x.mask, x.T)
    for rank in range(world):
        loss, gh, gW, t, seeds = res[rank]
        assert loss == pytest.approx(full["loss"], rel=1e-12)
        np.testing.assert_allclose(gW, full["grad_W"], rtol=1e-10, atol=1e-15)
        assert t == 11.0  # the slowest rank's time on every rank
        assert seeds == [3, 1003] and len(set(seeds)) == world
    np.testing.assert_allclose(np.concatenate([res[0][1], res[1][1]]), full["grad_h"],
                               rtol=1e-10, atol=1e-15)


def test_single_process_keeps_the_workload_seed():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.shard_seed(3, 0, 1) == 3
    assert bench.max_over_ranks(7.5, 1, "cpu") == 7.5
