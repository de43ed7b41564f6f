"""Pins of the fp64 top-K cache oracle (oracle/topk_cache_oracle.py) to things
other than itself: a brute-force selection written as plain loops, torch.topk
on distinct values, a worked example with ties, and properties of the
definition (permutation, shift and scale of the logits, K = V, NaN last).
Each pin would catch a plausible slip: reversed tie order, ascending order,
a NaN ranked first, an off-by-one in K, a transposed product."""
import numpy as np
import pytest
import torch

import oracle


def brute_force_topk(h, W, K):
    """Selection by repeated extraction of the best remaining entry, compared
    with explicit if-statements (larger logit wins; on equal logits the lower
    index wins; a NaN loses to any number, and to a NaN of lower index)."""
    N, d = len(h), len(h[0])
    V = len(W)
    out_i, out_v = [], []
    for r in range(N):
        z = []
        for v in range(V):
            s = 0.0
            for k in range(d):
                s += float(h[r][k]) * float(W[v][k])
            z.append(s)
        left = list(range(V))
        sel = []
        for _ in range(K):
            best = left[0]
            for v in left[1:]:
                a, b = z[v], z[best]
                if np.isnan(a):
                    better = np.isnan(b) and v < best
                elif np.isnan(b):
                    better = True
                else:
                    better = a > b or (a == b and v < best)
                if better:
                    best = v
            sel.append(best)
            left.remove(best)
        out_i.append(sel)
        out_v.append([z[v] for v in sel])
    return np.array(out_i), np.array(out_v)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    # small integers: many exactly equal logits
    h = rng.integers(-2, 3, size=(6, 4)).astype(np.float64)
    W = rng.integers(-2, 3, size=(23, 4)).astype(np.float64)
    for K in (1, 5, 23):
        i, v = oracle.topk_cache(h, W, K, block_rows=4)
        bi, bv = brute_force_topk(h.tolist(), W.tolist(), K)
        np.testing.assert_array_equal(i, bi)
        np.testing.assert_array_equal(v, bv)


def test_worked_example_with_ties():
    # z = h W^T = [1, 2, 1, 2, 0, 2]: three entries tie at 2 and two at 1
    W = np.array([[1, 0], [2, 0], [1, 0], [2, 0], [0, 0], [2, 5]], dtype=np.float64)
    h = np.array([[1, 0]], dtype=np.float64)
    i, v = oracle.topk_cache(h, W, 4)
    assert i.tolist() == [[1, 3, 5, 0]]
    assert v.tolist() == [[2.0, 2.0, 2.0, 1.0]]


def test_matches_torch_topk_on_distinct_values():
    rng = np.random.default_rng(7)
    h = rng.standard_normal((40, 16))
    W = rng.standard_normal((300, 16))
    i, v = oracle.topk_cache(h, W, 25, block_rows=16)
    tv, ti = torch.topk(torch.from_numpy(h) @ torch.from_numpy(W).T, 25, dim=1, sorted=True)
    np.testing.assert_array_equal(i, ti.numpy())
    np.testing.assert_allclose(v, tv.numpy(), rtol=1e-13, atol=1e-13)


def test_vocabulary_permutation_maps_indices():
    rng = np.random.default_rng(8)
    h = rng.standard_normal((10, 8))
    W = rng.standard_normal((50, 8))
    perm = rng.permutation(50)          # new row j holds old row perm[j]
    i, v = oracle.topk_cache(h, W, 12)
    pi, pv = oracle.topk_cache(h, W[perm], 12)
    np.testing.assert_array_equal(perm[pi], i)
    np.testing.assert_array_equal(pv, v)


def test_shift_and_positive_scale_keep_the_selection():
    rng = np.random.default_rng(9)
    h = rng.standard_normal((10, 8))
    W = rng.standard_normal((60, 8))
    i, v = oracle.topk_cache(h, W, 7)
    # a constant c_r added to every logit of row r: an extra input dimension
    c = rng.standard_normal((10, 1))
    i2, v2 = oracle.topk_cache(np.hstack([h, c]), np.hstack([W, np.ones((60, 1))]), 7)
    np.testing.assert_array_equal(i2, i)
    np.testing.assert_allclose(v2, v + c, rtol=1e-12, atol=1e-12)
    i3, v3 = oracle.topk_cache(3.0 * h, W, 7)
    np.testing.assert_array_equal(i3, i)
    np.testing.assert_allclose(v3, 3.0 * v, rtol=1e-12)


def test_k_equal_v_is_a_full_ranking():
    rng = np.random.default_rng(10)
    h = rng.standard_normal((3, 5))
    W = rng.standard_normal((31, 5))
    i, v = oracle.topk_cache(h, W, 31)
    for r in range(3):
        assert sorted(i[r].tolist()) == list(range(31))
        assert np.all(np.diff(v[r]) <= 0)


def test_row_logits_match_plain_loops_and_the_selected_values():
    # row_logits (used to check full-size cache rows one row at a time) is
    # the same product as the cache's logits: with small integers every dot
    # product is exact, so plain Python loops give the very same numbers, and
    # at the selected indices the rows hold the cache's own values
    rng = np.random.default_rng(11)
    h = rng.integers(-3, 4, size=(9, 6)).astype(np.float64)
    W = rng.integers(-3, 4, size=(41, 6)).astype(np.float64)
    rows = np.array([8, 0, 5, 5])
    Z = oracle.row_logits(h, W, rows)
    assert Z.shape == (4, 41)
    for i, r in enumerate(rows):
        for v in range(41):
            s = 0
            for k in range(6):
                s += int(h[r, k]) * int(W[v, k])
            assert Z[i, v] == s
    idx, val = oracle.topk_cache(h, W, 7)
    np.testing.assert_array_equal(np.take_along_axis(Z, idx[rows], axis=1), val[rows])


def test_nan_logits_rank_last():
    assert oracle.rank_order([1.0, np.nan, 5.0, np.nan, -np.inf]).tolist() == [2, 0, 4, 1, 3]
    with pytest.raises(ValueError):
        oracle.topk_cache(np.ones((1, 2)), np.ones((3, 2)), 4)


# ------------------------------------------------------------ planted mistakes

def _mutant_rank_order(kind):
    def rank(z_row):
        z = np.asarray(z_row, dtype=np.float64)
        v = np.arange(z.shape[0])
        nan = np.isnan(z)
        zz = np.where(nan, 0.0, z)
        if kind == "ties_high_index_first":
            return np.lexsort((-v, -zz, nan))
        if kind == "ascending":
            return np.lexsort((v, zz, nan))
        if kind == "nan_first":
            return np.lexsort((v, -zz, ~nan))
        if kind == "unstable_ties":
            return np.argsort(-zz, kind="quicksort")
        raise AssertionError(kind)
    return rank


PINS = [lambda: test_matches_brute_force_with_ties(0), test_worked_example_with_ties,
        test_matches_torch_topk_on_distinct_values, test_nan_logits_rank_last]


@pytest.mark.parametrize("kind", ["ties_high_index_first", "ascending", "nan_first",
                                  "unstable_ties"])
def test_planted_mistake_is_caught(kind, monkeypatch):
    from oracle import topk_cache_oracle as tco
    monkeypatch.setattr(tco, "rank_order", _mutant_rank_order(kind))
    monkeypatch.setattr(oracle, "rank_order", tco.rank_order)
    failed = False
    for p in PINS:
        try:
            p()
        except AssertionError:
            failed = True
            break
    assert failed, kind


def test_planted_off_by_one_in_k_is_caught(monkeypatch):
    from oracle import topk_cache_oracle as tco
    real = tco.topk_cache

    def short(h, W, K, block_rows=256):
        i, v = real(h, W, K, block_rows)
        i[:, -1] = i[:, 0]
        return i, v
    monkeypatch.setattr(oracle, "topk_cache", short)
    with pytest.raises(AssertionError):
        test_worked_example_with_ties()
