"""kd_topk_kl_fwd_bwd_noalloc, the entry point for callers that cannot
allocate device memory (a process whose memory pool owns the device, a plug-in
that is handed device pointers but no allocator).  It runs the same kernels as
kd_topk_kl_fwd_bwd with its workspace in a fixed scratch array that the
library holds, so its results must agree with the ordinary call and with the
fp64 oracle, and a second call must not be disturbed by what the first one left
in that shared array.

This file is named so that pytest collects it last."""
import numpy as np
import pytest

import oracle
import top_kl_loss_token_b300 as kd_mod
from top_kl_loss_token_b300 import synth
from kd_testutil import TOL, max_rel_err, to_device


def test_noalloc_rejects_sizes_beyond_the_scratch_array():
    # Host-side checks only: these return before any CUDA call, so they run
    # without a GPU.  Dummy (never dereferenced) pointers stand in for buffers.
    lib = kd_mod.load_library()
    p = 256
    call = lib.kd_topk_kl_fwd_bwd_noalloc
    # 1M tokens x K = 100: the sorted teacher lists alone need 800 MB.
    assert call(p, p, kd_mod.KD_BF16, p, p, None, 1 << 20, 4096, 201088, 100, 1.0, 0,
                p, p, p, None, None) == 3
    # fits at a small chunk, but not at the 4096-token chunk asked for
    assert kd_mod.workspace_bytes(4096, 256, 32000, 16, 128) <= kd_mod.KD_NOALLOC_SCRATCH_BYTES
    assert kd_mod.workspace_bytes(4096, 256, 32000, 16, 4096) > kd_mod.KD_NOALLOC_SCRATCH_BYTES
    assert call(p, p, kd_mod.KD_BF16, p, p, None, 4096, 256, 32000, 16, 1.0, 4096,
                p, p, p, None, None) == 3
    # invalid sizes keep the ordinary call's status codes
    assert call(p, p, kd_mod.KD_BF16, p, p, None, 64, 12, 512, 8, 1.0, 0, p, p, p, None, None) == 2
    assert call(p, p, kd_mod.KD_BF16, p, p, None, 64, 16, 0, 8, 1.0, 0, p, p, p, None, None) == 1


def _reference_and_noalloc(kd, x, chunk):
    import torch
    h, W, idx, lg, mask = to_device(x)
    err_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
    loss_r, gh_r, gW_r, _ = kd.fwd_bwd(h, W, idx, lg, mask, x.T, chunk, err_flags=err_ref)
    # outputs prepared by the caller; the call itself allocates nothing
    loss = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    gh = torch.full((x.N, x.d), float("nan"), dtype=torch.float32, device="cuda")
    gW = torch.full((x.V, x.d), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kd.fwd_bwd_noalloc(h, W, idx, lg, loss, gh, gW, mask, x.T, chunk, err_flags=err)
    torch.cuda.synchronize()
    assert int(err_ref.item()) == 0 and int(err.item()) == 0
    return ((loss_r.item(), gh_r.cpu().numpy(), gW_r.cpu().numpy()),
            (loss.item(), gh.cpu().numpy(), gW.cpu().numpy()))


def _assert_close(ref, got, dtype):
    tl, tg = TOL[dtype]
    assert abs(got[0] - ref[0]) <= tl * abs(ref[0]), (got[0], ref[0])
    assert np.isfinite(got[1]).all() and np.isfinite(got[2]).all()
    assert max_rel_err(got[1], ref[1]) <= tg
    assert max_rel_err(got[2], ref[2]) <= tg


def _assert_oracle(x, got):
    """The no-alloc results against the fp64 dense definition."""
    r = oracle.fwd_bwd(x.h_f32(), x.W_f32(), x.idx, x.logit, x.mask, x.T)
    _assert_close((r["loss"], r["grad_h"], r["grad_W"]), got, x.dtype)


@pytest.mark.gpu
def test_noalloc_matches_fwd_bwd_on_two_calls_in_a_row(kd):
    # first call: ragged vocabulary (3000 = 23.4 blocks of 128), 5 row tiles,
    # 15 % masked rows, the chunk picked by the call itself
    a = synth.make_inputs(640, 256, 3000, 16, T=2.0, dtype="bf16", seed=211, mask="random0.15")
    ref_a, got_a = _reference_and_noalloc(kd, a, 0)
    _assert_close(ref_a, got_a, "bf16")
    _assert_oracle(a, got_a)
    # second call, straight after, on the same scratch array: other sizes, no
    # mask, three chunks of 128 tokens with a short last one
    b = synth.make_inputs(300, 128, 1000, 8, T=1.0, dtype="bf16", seed=212)
    ref_b, got_b = _reference_and_noalloc(kd, b, 128)
    _assert_close(ref_b, got_b, "bf16")
    _assert_oracle(b, got_b)
