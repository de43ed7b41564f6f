"""GPU parity of the CUDA path against the fp64 oracle, element by element, at
sizes the oracle finishes in seconds that still span several tiles, several
chunks and ragged tails; plus the edge cases the method has."""
import numpy as np
import pytest

import oracle
from top_kl_loss_token_b300 import synth
from kd_testutil import TOL, assert_parity, max_rel_err, run_gpu, to_device

pytestmark = pytest.mark.gpu


def oracle_of(x):
    return oracle.fwd_bwd(x.h_f32(), x.W_f32(), x.idx, x.logit, x.mask, x.T)


def check_full(kd, x, chunk=0):
    ref = oracle_of(x)
    got = run_gpu(kd, x, chunk)
    assert got["n_valid"] == ref["n_valid"]
    errs = assert_parity(got, ref, x.dtype)
    valid_rows = np.nonzero(ref["valid"])[0]
    np.testing.assert_array_equal(got["rows"], valid_rows)
    tl = TOL[x.dtype][0]
    np.testing.assert_allclose(got["lse"], ref["lse"][valid_rows], rtol=tl, atol=tl)
    np.testing.assert_allclose(got["loss_rows"], ref["loss_rows"][valid_rows], rtol=10 * tl,
                               atol=10 * tl * max(1.0, abs(ref["loss"])))
    return got, ref, errs


# ------------------------------------------------------------ tensor-core GEMM

@pytest.mark.parametrize("a_mn", [0, 1])
@pytest.mark.parametrize("b_mn", [0, 1])
@pytest.mark.parametrize("M,N,K", [(200, 296, 136), (256, 512, 1000), (2048, 5120, 128)])
def test_umma_gemm_operand_layouts(kd, a_mn, b_mn, M, N, K):
    import torch
    g = torch.Generator().manual_seed(M * 7 + N * 3 + K + 11 * a_mn + 5 * b_mn)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g).to(torch.bfloat16)
    want = A.double() @ B.double().T
    Ad = (A.T.contiguous() if a_mn else A).cuda()
    Bd = (B.T.contiguous() if b_mn else B).cuda()
    out, err = kd.kd_umma_gemm_bf16(Ad, Bd, M, N, K, a_mn, b_mn)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = out.cpu().double()
    assert float((got - want).abs().max()) <= 2e-5 * float(want.abs().max()) + 1e-4
    # accumulate: D += A B^T
    out2, err = kd.kd_umma_gemm_bf16(Ad, Bd, M, N, K, a_mn, b_mn, out=out.clone(), accumulate=True)
    torch.cuda.synchronize()
    assert float((out2.cpu().double() - 2 * want).abs().max()) <= 4e-5 * float(want.abs().max()) + 2e-4


# ------------------------------------------------------------ end to end, bf16

@pytest.mark.parametrize("chunk", [0, 256, 1000])
def test_parity_bf16_masked_ragged(kd, chunk):
    # V = 3000 is 23.4 column blocks of 128, N = 600 spans 5 row tiles of 128
    # and, at chunk 256, three chunks with a short last one.
    x = synth.make_inputs(600, 256, 3000, 16, T=2.0, dtype="bf16", seed=101, mask="random0.2")
    check_full(kd, x, chunk)


def test_parity_bf16_unmasked(kd):
    x = synth.make_inputs(300, 128, 1000, 5, T=1.0, dtype="bf16", seed=102)
    check_full(kd, x)


def test_parity_bf16_packed_heavy_head(kd):
    x = synth.make_inputs(1024, 512, 4096, 100, T=2.0, dtype="bf16", seed=103, heavy_head=True,
                          mask="packed", B=2, doc=(80, 230), pad=(2, 30))
    check_full(kd, x, chunk=384)


def test_chunk_invariance(kd):
    x = synth.make_inputs(700, 192, 2500, 12, T=1.0, dtype="bf16", seed=104, mask="random0.1")
    a = run_gpu(kd, x, 128)
    b = run_gpu(kd, x, 700)
    c = run_gpu(kd, x, 333)
    for o in (b, c):
        assert abs(o["loss"] - a["loss"]) <= 1e-5 * abs(a["loss"])
        assert max_rel_err(o["grad_h"], a["grad_h"]) <= 2e-3
        assert max_rel_err(o["grad_W"], a["grad_W"]) <= 2e-3


def test_fwd_only_matches(kd):
    x = synth.make_inputs(400, 128, 1500, 8, T=1.5, dtype="bf16", seed=105, mask="random0.3")
    a = run_gpu(kd, x, 200)
    b = run_gpu(kd, x, 200, want_grads=False)
    assert b["loss"] == pytest.approx(a["loss"], rel=1e-6)
    ref = oracle.fwd(x.h_f32(), x.W_f32(), x.idx, x.logit, x.mask, x.T)
    assert b["loss"] == pytest.approx(ref["loss"], rel=TOL["bf16"][0])


# ------------------------------------------------------------ fp32 CUDA-core path

def test_fp32_tiny_config(kd):
    x = synth.make_config(1)
    check_full(kd, x)


def test_fp32_masked_ragged(kd):
    x = synth.make_inputs(150, 20, 300, 7, T=2.0, dtype="fp32", seed=106, mask="random0.25",
                          w_std=0.3)
    check_full(kd, x, chunk=64)


# ------------------------------------------------------------ edge cases

def test_empty_input(kd):
    import torch
    d, V, K = 64, 300, 4
    h = torch.zeros(0, d, dtype=torch.bfloat16, device="cuda")
    W = torch.randn(V, d, device="cuda").to(torch.bfloat16)
    idx = torch.zeros(0, K, dtype=torch.int32, device="cuda")
    lg = torch.zeros(0, K, dtype=torch.float32, device="cuda")
    loss, gh, gW, _ = kd.fwd_bwd(h, W, idx, lg, None, 1.0)
    torch.cuda.synchronize()
    assert loss.item() == 0.0 and gh.numel() == 0 and float(gW.abs().max()) == 0.0


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_all_rows_masked(kd, dtype):
    x = synth.make_inputs(90, 64, 700, 6, dtype=dtype, seed=107)
    x.mask = np.zeros(90, np.uint8)
    got = run_gpu(kd, x, 64)
    assert got["loss"] == 0.0 and got["n_valid"] == 0
    assert np.all(got["grad_h"] == 0) and np.all(got["grad_W"] == 0)


def test_single_entry_and_duplicate_indices(kd):
    x = synth.make_inputs(200, 64, 800, 1, T=1.0, dtype="bf16", seed=108)
    check_full(kd, x)
    y = synth.make_inputs(200, 64, 40, 30, T=1.0, dtype="bf16", seed=109)
    rng = np.random.default_rng(0)
    y.idx = rng.integers(0, 40, size=y.idx.shape).astype(np.int32)  # many duplicates
    check_full(kd, y)


def test_full_vocabulary_teacher(kd):
    # K = V: the top-K loss becomes the full KL.
    x = synth.make_inputs(130, 64, 384, 384, T=1.0, dtype="bf16", seed=110)
    x.idx = np.stack([np.random.default_rng(i).permutation(384) for i in range(130)]).astype(np.int32)
    check_full(kd, x)


def test_zero_loss_when_teacher_equals_student(kd):
    # d = V = K = 64, W = I: z = h exactly; teacher logits = h at idx -> KL = 0.
    V = d = 64
    N = 256
    rng = np.random.default_rng(5)
    hv = (np.round(rng.normal(size=(N, d)) * 4) / 4).astype(np.float32)
    idx = np.stack([rng.permutation(V) for _ in range(N)]).astype(np.int32)
    x = synth.KDInputs("eq", "bf16", synth.bf16_bits(hv), synth.bf16_bits(np.eye(V, dtype=np.float32)),
                       idx, np.take_along_axis(hv, idx, axis=1).astype(np.float32), None, 1.0, 0)
    got = run_gpu(kd, x)
    # The stored exponentials are bf16 (relative error up to 2^-8), so the
    # gradient is zero up to about 2^-8 of a typical entry 1 / (T N) = 0.004.
    assert abs(got["loss"]) < 1e-4
    assert np.abs(got["grad_h"]).max() < 2e-5 and np.abs(got["grad_W"]).max() < 2e-5


def test_out_of_range_and_bad_teacher_rows(kd):
    x = synth.make_inputs(260, 64, 900, 10, T=1.0, dtype="bf16", seed=111, mask="random0.1")
    x.mask[[3, 7, 11, 12, 13, 14]] = 1
    x.idx[3, 2] = 900
    x.idx[7, 0] = -5
    x.logit[11, 4] = np.nan
    x.logit[12, :] = -np.inf
    x.logit[13, 1] = np.inf
    x.logit[14, 5] = -np.inf
    got, ref, _ = check_full(kd, x, chunk=128)
    assert ref["flags"] == (oracle.FLAG_INDEX_RANGE | oracle.FLAG_BAD_TEACHER)
    assert got["err"] == ref["flags"]


def test_masked_rows_data_is_never_read(kd):
    x = synth.make_inputs(300, 64, 700, 6, T=1.0, dtype="bf16", seed=112, mask="random0.3")
    clean = run_gpu(kd, x, 128)
    bad = np.nonzero(x.mask == 0)[0]
    x.h[bad] = 0x7FC0     # bf16 NaN
    x.logit[bad] = np.nan
    x.idx[bad] = 10 ** 6
    dirty = run_gpu(kd, x, 128)
    assert dirty["err"] == 0
    assert dirty["loss"] == clean["loss"]
    np.testing.assert_array_equal(dirty["grad_h"], clean["grad_h"])
    np.testing.assert_array_equal(dirty["grad_W"], clean["grad_W"])
