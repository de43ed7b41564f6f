"""The data-parallel split on one GPU: the batch's tokens are cut into shards
(as ranks would own them), every shard is prepared on its own
(kd_topk_kl_prepare), the shards' counts are summed, and every shard runs the
chunk loop with the batch's count as divisor (kd_topk_kl_fwd_bwd_prepared).
The shards' losses and grad_W add up to the batch's and their grad_h rows are
the batch's rows: checked against the fp64 oracle on the whole batch and
against one kd_topk_kl_fwd_bwd call over it.  The shards run one after the
other on one stream (no kernel waits on another)."""
import numpy as np
import pytest

import oracle
from top_kl_loss_token_b300 import synth
from kd_testutil import TOL, max_rel_err, run_gpu, to_device

pytestmark = pytest.mark.gpu


def _shards(kd, x, cuts, chunk):
    import torch
    h, W, idx, lg, mask = to_device(x)
    dt = kd.KD_BF16 if x.dtype == "bf16" else kd.KD_FP32
    bounds = [0, *cuts, x.N]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    preps = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        m = None if mask is None else mask[a:b]
        n, ws = kd.prepare(idx[a:b], lg[a:b], m, b - a, x.d, x.V, x.T, chunk, dt, err_flags=err)
        preps.append((a, b, n, ws))
    total = torch.zeros(1, dtype=torch.int64, device="cuda")
    for _, _, n, _ in preps:
        total += n  # what an all-reduce of the counts computes
    outs = []
    for a, b, n, ws in preps:
        loss, gh, gW = kd.fwd_bwd_prepared(h[a:b], W, x.K, ws, n_norm=total, T=x.T, chunk=chunk,
                                           err_flags=err)
        outs.append((loss, gh, gW, n))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    loss = sum(float(o[0].item()) for o in outs)
    gW = sum(o[2].double() for o in outs).cpu().numpy()
    gh = torch.cat([o[1] for o in outs]).cpu().numpy().astype(np.float64)
    counts = [int(o[3].item()) for o in outs]
    return loss, gh, gW, counts, int(total.item())


@pytest.mark.parametrize("dtype,cuts,chunk", [("bf16", [300, 301], 128), ("bf16", [257], 0),
                                              ("fp32", [100, 333], 96)])
def test_shards_with_the_batch_divisor_match_the_whole_batch(kd, dtype, cuts, chunk):
    x = synth.make_inputs(700, 128, 3000, 16, T=2.0, dtype=dtype, seed=61, mask="random0.2",
                          w_std=0.05 if dtype == "bf16" else 0.1)
    loss, gh, gW, counts, total = _shards(kd, x, cuts, chunk)
    ref = oracle.fwd_bwd(x.h_f32(), x.W_f32(), x.idx, x.logit, x.mask, x.T)
    assert total == ref["n_valid"] and sum(counts) == total
    bounds = [0, *cuts, x.N]
    assert counts == [int(x.mask[a:b].sum()) for a, b in zip(bounds[:-1], bounds[1:])]
    tl, tg = TOL[dtype]
    assert abs(loss - ref["loss"]) <= tl * abs(ref["loss"])
    assert max_rel_err(gh, ref["grad_h"]) <= tg
    assert max_rel_err(gW, ref["grad_W"]) <= tg
    # and against one call over the whole batch: the same kernels on the same
    # rows, so grad_h matches to the rounding of the chunk boundaries only
    one = run_gpu(kd, x, chunk=chunk)
    assert abs(loss - one["loss"]) <= tl * abs(one["loss"])
    assert max_rel_err(gh, one["grad_h"]) <= tg
    assert max_rel_err(gW, one["grad_W"]) <= tg


def test_prepare_then_prepared_with_the_own_count_is_fwd_bwd(kd):
    # n_norm = this call's own count (or NULL) is kd_topk_kl_fwd_bwd, bit for bit
    import torch
    x = synth.make_inputs(520, 256, 4000, 32, T=1.0, dtype="bf16", seed=62, mask="random0.1")
    h, W, idx, lg, mask = to_device(x)
    a = run_gpu(kd, x, chunk=256, tensors=(h, W, idx, lg, mask))
    n, ws = kd.prepare(idx, lg, mask, x.N, x.d, x.V, x.T, 256, kd.KD_BF16)
    l1, gh1, gW1 = kd.fwd_bwd_prepared(h, W, x.K, ws, n_norm=n, T=x.T, chunk=256)
    n2, ws2 = kd.prepare(idx, lg, mask, x.N, x.d, x.V, x.T, 256, kd.KD_BF16)
    l2, gh2, gW2 = kd.fwd_bwd_prepared(h, W, x.K, ws2, n_norm=None, T=x.T, chunk=256)
    lf = kd.fwd_prepared(h, W, x.K, ws2, n_norm=n2, T=x.T, chunk=256)
    torch.cuda.synchronize()
    assert int(n.item()) == a["n_valid"] == int(x.mask.sum())
    for loss, gh, gW in ((l1, gh1, gW1), (l2, gh2, gW2)):
        assert float(loss.item()) == a["loss"]
        assert np.array_equal(gh.cpu().numpy(), a["grad_h"].astype(np.float32))
        assert np.array_equal(gW.cpu().numpy(), a["grad_W"].astype(np.float32))
    assert float(lf.item()) == pytest.approx(a["loss"], rel=1e-6)


def test_fwd_bwd_dp_on_one_rank_is_fwd_bwd(kd):
    import torch
    x = synth.make_inputs(300, 128, 2000, 8, T=1.0, dtype="bf16", seed=63)
    h, W, idx, lg, mask = to_device(x)
    a = run_gpu(kd, x, tensors=(h, W, idx, lg, mask))
    loss, gh, gW, n, _ = kd.fwd_bwd_dp(h, W, idx, lg, mask, x.T)
    torch.cuda.synchronize()
    assert int(n.item()) == x.N
    assert float(loss.item()) == a["loss"]
    assert np.array_equal(gW.cpu().numpy(), a["grad_W"].astype(np.float32))


def test_zero_divisor_gives_zero(kd):
    import torch
    x = synth.make_inputs(200, 64, 1000, 8, T=1.0, dtype="bf16", seed=64)
    h, W, idx, lg, mask = to_device(x)
    n, ws = kd.prepare(idx, lg, mask, x.N, x.d, x.V, x.T, 0, kd.KD_BF16)
    zero = torch.zeros(1, dtype=torch.int64, device="cuda")
    loss, gh, gW = kd.fwd_bwd_prepared(h, W, x.K, ws, n_norm=zero, T=x.T)
    torch.cuda.synchronize()
    assert float(loss.item()) == 0.0
    assert not gh.abs().max().item() and not gW.abs().max().item()
