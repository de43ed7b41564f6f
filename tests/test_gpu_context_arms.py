"""The two plain-PyTorch baselines that bench.py --dense-context runs beside
the fused call for the pages' memory comparison (ai2day.live story, the
comparison table: dense KL, forward-chunked KL, the fused chunked loss) must
compute the same loss and gradients: each is checked against the fp64 oracle
and against kd_topk_kl_fwd_bwd on a few hundred tokens, at the bf16
tolerances (the arms keep bf16 logits and gradients)."""
import os
import sys

import numpy as np
import pytest

import oracle
from top_kl_loss_token_b300 import synth
from kd_testutil import TOL, max_rel_err, run_gpu, to_device

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
@pytest.mark.parametrize("arm_chunk", [0, 128])
def test_context_arm_matches_the_oracle_and_the_fused_call(kd, arm_chunk):
    sys.path.insert(0, ROOT)
    import bench
    x = synth.make_inputs(384, 128, 3000, 16, T=1.5, dtype="bf16", seed=71, w_std=0.05)
    h, W, idx, lg, _ = to_device(x)
    loss, gh, gW = bench.torch_kl_arm(h, W, idx, lg, x.T, arm_chunk)
    ref = oracle.fwd_bwd(x.h_f32(), x.W_f32(), x.idx, x.logit, None, x.T)
    tl, tg = TOL["bf16"]
    assert abs(float(loss) - ref["loss"]) <= tl * abs(ref["loss"])
    assert max_rel_err(gh.double().cpu().numpy(), ref["grad_h"]) <= tg
    assert max_rel_err(gW.double().cpu().numpy(), ref["grad_W"]) <= tg
    fused = run_gpu(kd, x, tensors=(h, W, idx, lg, None))
    assert abs(float(loss) - fused["loss"]) <= tl * abs(fused["loss"])
    assert max_rel_err(gh.double().cpu().numpy(), fused["grad_h"]) <= tg
    assert max_rel_err(gW.double().cpu().numpy(), fused["grad_W"]) <= tg


@pytest.mark.parametrize("arm_chunk", [0, 50])
def test_context_arm_arithmetic_on_cpu(arm_chunk):
    # the same arms on the CPU with fp32 inputs, at the fp32 tolerances
    sys.path.insert(0, ROOT)
    import torch
    import bench
    x = synth.make_inputs(120, 32, 400, 8, T=2.0, dtype="fp32", seed=72, w_std=0.2)
    loss, gh, gW = bench.torch_kl_arm(torch.from_numpy(x.h), torch.from_numpy(x.W),
                                      torch.from_numpy(x.idx), torch.from_numpy(x.logit), x.T,
                                      arm_chunk)
    ref = oracle.fwd_bwd(x.h_f32(), x.W_f32(), x.idx, x.logit, None, x.T)
    tl, tg = TOL["fp32"]
    assert abs(float(loss) - ref["loss"]) <= tl * abs(ref["loss"])
    assert max_rel_err(gh.double().numpy(), ref["grad_h"]) <= tg
    assert max_rel_err(gW.double().numpy(), ref["grad_W"]) <= tg
