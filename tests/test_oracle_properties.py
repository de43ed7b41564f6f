"""Randomised properties of the fp64 loss oracle (hypothesis draws the sizes,
temperature, mask and data): facts the definition fixes for every input, each
checked without recomputing the oracle's own formula.

  - Gibbs: with distinct indices every valid row's KL term is >= 0;
  - the gradient sum rule: every row of dL/dz sums to zero, so the column
    sums of grad_W vanish;
  - masking a row is deleting it (N_valid and the mean follow);
  - permuting the K entries of each row changes nothing;
  - the blocking over rows changes nothing beyond rounding;
  - the temperature identity loss_T(h, l) = loss_1(h / T, l / T).
"""
import numpy as np
import pytest
from hypothesis import given, settings
from hypothesis import strategies as st

import oracle

SETTINGS = dict(max_examples=40, deadline=None, derandomize=True)


@st.composite
def problems(draw):
    N = draw(st.integers(1, 9))
    d = draw(st.integers(1, 6))
    V = draw(st.integers(2, 40))
    K = draw(st.integers(1, min(V, 8)))
    T = draw(st.sampled_from([0.5, 1.0, 2.0, 3.0]))
    seed = draw(st.integers(0, 2 ** 31 - 1))
    rng = np.random.default_rng(seed)
    h = rng.normal(size=(N, d)) * draw(st.sampled_from([0.3, 1.0, 3.0]))
    W = rng.normal(size=(V, d))
    idx = np.stack([rng.permutation(V)[:K] for _ in range(N)]).astype(np.int32)
    logit = rng.normal(size=(N, K)) * 2.0
    mask = (rng.random(N) < 0.8).astype(np.uint8)
    mask[rng.integers(0, N)] = 1
    return h, W, idx, logit, mask, T


@settings(**SETTINGS)
@given(problems())
def test_gibbs_and_sum_rule(prob):
    h, W, idx, logit, mask, T = prob
    r = oracle.fwd_bwd(h, W, idx, logit, mask, T)
    assert np.all(r["loss_rows"][r["valid"]] >= -1e-12)
    assert r["loss"] >= -1e-12
    scale = max(1.0, float(np.abs(r["grad_W"]).max()))
    assert np.abs(r["grad_W"].sum(axis=0)).max() <= 1e-12 * scale * max(1, h.shape[0])


@settings(**SETTINGS)
@given(problems())
def test_masking_is_deletion(prob):
    h, W, idx, logit, mask, T = prob
    r = oracle.fwd_bwd(h, W, idx, logit, mask, T)
    keep = mask != 0
    s = oracle.fwd_bwd(h[keep], W, idx[keep], logit[keep], None, T)
    assert r["n_valid"] == s["n_valid"] == int(keep.sum())
    assert r["loss"] == pytest.approx(s["loss"], rel=1e-12, abs=1e-15)
    np.testing.assert_allclose(r["grad_W"], s["grad_W"], rtol=1e-10, atol=1e-15)
    np.testing.assert_allclose(r["grad_h"][keep], s["grad_h"], rtol=1e-10, atol=1e-15)
    assert np.all(r["grad_h"][~keep] == 0)


@settings(**SETTINGS)
@given(problems(), st.integers(0, 2 ** 31 - 1))
def test_entry_order_and_row_blocking(prob, seed):
    h, W, idx, logit, mask, T = prob
    rng = np.random.default_rng(seed)
    perm = np.stack([rng.permutation(idx.shape[1]) for _ in range(idx.shape[0])])
    a = oracle.fwd_bwd(h, W, idx, logit, mask, T)
    b = oracle.fwd_bwd(h, W, np.take_along_axis(idx, perm, 1), np.take_along_axis(logit, perm, 1),
                       mask, T, block_rows=2)
    assert a["loss"] == pytest.approx(b["loss"], rel=1e-12, abs=1e-15)
    np.testing.assert_allclose(a["grad_h"], b["grad_h"], rtol=1e-10, atol=1e-15)
    np.testing.assert_allclose(a["grad_W"], b["grad_W"], rtol=1e-10, atol=1e-15)


@settings(**SETTINGS)
@given(problems())
def test_temperature_identity(prob):
    h, W, idx, logit, mask, T = prob
    a = oracle.fwd_bwd(h, W, idx, logit, mask, T)
    b = oracle.fwd_bwd(h / T, W, idx, logit / T, mask, 1.0)
    assert a["loss"] == pytest.approx(b["loss"], rel=1e-10, abs=1e-14)
    # d/dh at temperature T is (1/T) times d/d(h/T) at temperature 1
    np.testing.assert_allclose(a["grad_h"], b["grad_h"] / T, rtol=1e-9, atol=1e-14)
