"""The token-sharded (data-parallel) path on CPU with two gloo ranks.

The loss shards by tokens: each rank runs the fused loss on its own tokens
with W replicated.  The batch's loss is the mean over all of its valid tokens,
so the library splits a step in two (kd_topk_kl_prepare, then the chunk loop
with a divisor): each rank counts its valid rows, the counts are all-reduced,
every rank divides by the batch's count, and loss and grad_W are all-reduced
(fwd_bwd_dp).  Here the two library calls are replaced by the fp64 oracle on
the rank's shard (the GPU kernels are checked against that oracle elsewhere),
so the test runs fwd_bwd_dp's own exchange logic under torch.distributed and
checks it against the oracle on the whole batch.  The bench's rank logic (one
seed per shard, the slowest rank's time) is checked on the same two ranks."""
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


def _problem():
    from top_kl_loss_token_b300 import synth
    return synth.make_inputs(90, 32, 300, 6, T=2.0, dtype="fp32", seed=5, mask="random0.3",
                             w_std=0.3)


def _oracle_backed_library(kd, oracle, x, sl, seen):
    """Stand-ins for the two library calls of fwd_bwd_dp, computed by the
    oracle on this rank's shard; they record the divisor they were given."""
    h = x.h_f32()[sl]
    m = x.mask[sl]

    def validate(h_, W_, idx_, lg_, mask_):
        return h_.shape[0], h_.shape[1], W_.shape[0], idx_.shape[1]

    def prepare(topk_idx, topk_logit, mask, N, d, V, T=1.0, chunk=0, dtype=0, workspace=None,
                n_valid=None, err_flags=None, stream=None):
        p, valid, _ = oracle.teacher_distribution(x.idx[sl], x.logit[sl], m, V, T)
        return torch.tensor([int(valid.sum())], dtype=torch.int64), {"prepared": True}

    def prepared(h_, W_, K, workspace, n_norm=None, T=1.0, chunk=0, loss=None, grad_h=None,
                 grad_W=None, err_flags=None, stream=None):
        assert workspace == {"prepared": True}
        seen.append(int(n_norm.item()))
        r = oracle.fwd_bwd(h, x.W_f32(), x.idx[sl], x.logit[sl], m, T, n_norm=int(n_norm.item()))
        return (torch.tensor([r["loss"]], dtype=torch.float64), torch.from_numpy(r["grad_h"]),
                torch.from_numpy(r["grad_W"].copy()))

    kd._validate = validate
    kd._dtype_code = lambda t: kd.KD_FP32
    kd.kd_topk_kl_prepare = prepare
    kd.kd_topk_kl_fwd_bwd_prepared = prepared


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    import top_kl_loss_token_b300 as kd
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x = _problem()
        # uneven shards with different valid counts
        cut = 37
        sl = slice(0, cut) if rank == 0 else slice(cut, x.N)
        seen = []
        _oracle_backed_library(kd, oracle, x, sl, seen)
        h = torch.from_numpy(x.h_f32()[sl])
        W = torch.from_numpy(x.W_f32())
        loss, gh, gW, n_total, _ = kd.fwd_bwd_dp(h, W, torch.from_numpy(x.idx[sl]),
                                                torch.from_numpy(x.logit[sl]),
                                                torch.from_numpy(x.mask[sl]), x.T)
        # bench rank logic
        t = bench.max_over_ranks(10.0 + rank, world, "cpu")
        seeds = [bench.shard_seed(3, k, world) for k in range(world)]
        q.put((rank, float(loss.item()), gh.numpy(), gW.numpy(), int(n_total.item()), seen, t,
               seeds))
    finally:
        dist.destroy_process_group()


def test_token_sharded_step_matches_whole_batch():
    import oracle
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        rank, *rest = q.get(timeout=120)
        res[rank] = rest
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    x = _problem()
    full = oracle.fwd_bwd(x.h_f32(), x.W_f32(), x.idx, x.logit, x.mask, x.T)
    for rank in range(world):
        loss, gh, gW, n_total, seen, t, seeds = res[rank]
        # every rank divided by the batch's count, not its own
        assert n_total == full["n_valid"] and seen == [full["n_valid"]]
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
