"""GPU parity of the teacher top-K cache builder (kd_topk_cache_build) with
the fp64 oracle (oracle/topk_cache_oracle.py).

With small-integer inputs every product and partial sum is exact in fp32, so
the kernel's logits equal the oracle's exactly and the ranking -- including
the many ties such inputs create -- must match index for index and bit for
bit.  With Gaussian inputs the fp32 accumulation order decides near-ties, so
there the unique parts are compared (values at the chosen indices, the order)
and any index that differs from the oracle's must be a near-tie of the K-th
value."""
import numpy as np
import pytest

import oracle
from top_kl_loss_token_b300 import synth

pytestmark = pytest.mark.gpu


def _bf16_tensor(a):
    import torch
    return torch.from_numpy(synth.bf16_bits(a).view(np.int16)).view(torch.bfloat16).cuda()


def _run(kd, h, W, K, chunk=0):
    import torch
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx, val, _ = kd.topk_cache_build(_bf16_tensor(h), _bf16_tensor(W), K, chunk, err_flags=err)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), val.cpu().numpy(), int(err.item())


def _int_inputs(seed, N, d, V, lo=-2, hi=3):
    rng = np.random.default_rng(seed)
    h = rng.integers(lo, hi, size=(N, d)).astype(np.float32)
    W = rng.integers(lo, hi, size=(V, d)).astype(np.float32)
    return h, W


@pytest.mark.parametrize("K,chunk", [(1, 0), (7, 128), (100, 0), (100, 256)])
def test_exact_integer_logits_with_ties(kd, K, chunk):
    # N = 300 spans two 256-row pair tiles, V = 3000 is 23.4 blocks of 128
    h, W = _int_inputs(1 + K, 300, 64, 3000)
    gi, gv, err = _run(kd, h, W, K, chunk)
    oi, ov = oracle.topk_cache(h, W, K)
    assert err == 0
    np.testing.assert_array_equal(gi, oi)
    np.testing.assert_array_equal(gv, ov.astype(np.float32))


@pytest.mark.parametrize("K", [200, 300])
def test_more_entries_than_blocks_and_full_ranking(kd, K):
    # V = 300 has 3 blocks of 128: K > 3, every logit is a candidate
    h, W = _int_inputs(7, 130, 32, 300)
    gi, gv, err = _run(kd, h, W, K)
    oi, ov = oracle.topk_cache(h, W, K)
    assert err == 0
    np.testing.assert_array_equal(gi, oi)
    np.testing.assert_array_equal(gv, ov.astype(np.float32))


def test_maximum_k(kd):
    # K = KD_MAX_K = 4096 of a 6000-word vocabulary (47 blocks of 128: every
    # logit is a candidate), exact on integer inputs
    h, W = _int_inputs(13, 130, 32, 6000)
    gi, gv, err = _run(kd, h, W, kd.KD_MAX_K)
    oi, ov = oracle.topk_cache(h, W, kd.KD_MAX_K)
    assert err == 0
    np.testing.assert_array_equal(gi, oi)
    np.testing.assert_array_equal(gv, ov.astype(np.float32))


def test_constant_rows_fill_the_candidate_bound(kd):
    # a zero hidden state gives equal logits everywhere: the K lowest indices,
    # and exactly 128 K candidates (the bound) in pass 2
    h, W = _int_inputs(8, 40, 32, 20000)
    h[3] = 0.0
    h[17] = 0.0
    gi, gv, err = _run(kd, h, W, 100)
    oi, ov = oracle.topk_cache(h, W, 100)
    assert err == 0
    np.testing.assert_array_equal(gi, oi)
    np.testing.assert_array_equal(gi[3], np.arange(100))
    np.testing.assert_array_equal(gv, ov.astype(np.float32))


@pytest.mark.parametrize("chunk", [0, 128])
def test_sampled_threshold_overflow_is_redone_exactly(kd, chunk):
    # V = 8192 is 64 blocks and K = 4, so the first threshold comes from the
    # first 8 blocks (1024 columns), where every logit is 0.  Rows with
    # h = 1 have logits >= 16 in all 7168 later columns: far more candidates
    # than the capacity of 128 K = 512, so they are redone with the tight
    # threshold.  Rows with h = -1 keep the sampled threshold (385
    # candidates), random rows fall either way; with 128-row chunks the
    # second chunk (all h = -1) has no overflowing row, so its third pass
    # returns at once.
    rng = np.random.default_rng(21)
    d, V, N, K = 16, 8192, 250, 4
    W = np.zeros((V, d), np.float32)
    W[1024:] = rng.integers(1, 4, size=(V - 1024, d))
    h = rng.integers(-2, 3, size=(N, d)).astype(np.float32)
    h[:40] = 1.0
    h[40:80] = -1.0
    h[128:] = -1.0
    gi, gv, err = _run(kd, h, W, K, chunk)
    oi, ov = oracle.topk_cache(h, W, K)
    assert err == 0
    np.testing.assert_array_equal(gi, oi)
    np.testing.assert_array_equal(gv, ov.astype(np.float32))
    np.testing.assert_array_equal(gi[50], np.arange(K))


def test_nan_hidden_state_ranks_last_and_is_flagged(kd):
    h, W = _int_inputs(9, 64, 32, 1000)
    h[5, 3] = np.nan
    gi, gv, err = _run(kd, h, W, 10)
    assert err & kd.KD_FLAG_BAD_TEACHER
    oi, ov = oracle.topk_cache(h, W, 10)
    np.testing.assert_array_equal(gi, oi)
    assert np.isnan(gv[5]).all() and gi[5].tolist() == list(range(10))
    ok = np.arange(64) != 5
    np.testing.assert_array_equal(gv[ok], ov[ok].astype(np.float32))


def _check_gaussian(h, W, K, gi, gv, rows=None):
    """Values at the chosen indices match fp64 within fp32 accumulation error,
    values are in rank order, and every index that differs from the oracle's
    selection is within that error of the oracle's K-th value."""
    rows = np.arange(h.shape[0]) if rows is None else rows
    Z = oracle.row_logits(h, W, rows)
    d = h.shape[1]
    for j, r in enumerate(rows):
        z = Z[j]
        tol = 4 * d * 2.0 ** -24 * float(np.abs(h[r]).max() * np.abs(W).max()) + 1e-6
        order = oracle.rank_order(z)[:K]
        np.testing.assert_allclose(gv[r], z[gi[r]], rtol=0, atol=tol)
        assert np.all(np.diff(gv[r]) <= 0)
        assert len(set(gi[r].tolist())) == K
        kth = z[order[-1]]
        for v in set(gi[r].tolist()) ^ set(order.tolist()):
            assert abs(z[v] - kth) <= 2 * tol, (r, v, z[v], kth)


def test_gaussian_inputs(kd):
    rng = np.random.default_rng(11)
    h = synth.bf16_bits_to_f32(synth.bf16_bits(rng.standard_normal((520, 256)).astype(np.float32)))
    W = synth.bf16_bits_to_f32(synth.bf16_bits(
        (0.02 * rng.standard_normal((5000, 256))).astype(np.float32)))
    gi, gv, err = _run(kd, h, W, 100, chunk=256)
    assert err == 0
    _check_gaussian(h, W, 100, gi, gv)


@pytest.mark.slow
def test_full_vocabulary_sampled_rows(kd):
    # the 201,088-entry vocabulary at d = 2880, rows checked one by one
    rng = np.random.default_rng(12)
    N, d, V = 2048, 2880, 201088
    h = synth.bf16_bits_to_f32(synth.bf16_bits(rng.standard_normal((N, d)).astype(np.float32)))
    W = synth.bf16_bits_to_f32(synth.bf16_bits(
        (0.02 * rng.standard_normal((V, d))).astype(np.float32)))
    gi, gv, err = _run(kd, h, W, 100)
    assert err == 0
    rows = np.concatenate([[0, N - 1], rng.choice(N, 30, replace=False)])
    _check_gaussian(h, W, 100, gi, gv, rows)
