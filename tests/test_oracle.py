"""Pins for the fp64 oracle, each against something other than the oracle itself:
closed forms, a case where the loss must vanish, Gibbs' inequality, library
routines (cross-entropy for K = 1, kl_div for K = V, autograd), central finite
differences, and the invariances the write-ups imply (the chunked loss being
"mathematically equivalent" to the dense one: iwenai.com essay, paragraph after
"Enter a new approach")."""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from top_kl_loss_token_b300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def rand_problem(N=6, d=5, V=11, K=3, T=1.0, seed=0, distinct=True, scale=1.0):
    rng = np.random.default_rng(seed)
    h = rng.normal(size=(N, d)) * scale
    W = rng.normal(size=(V, d)) * scale
    if distinct:
        idx = np.stack([rng.permutation(V)[:K] for _ in range(N)])
    else:
        idx = rng.integers(0, V, size=(N, K))
    logit = rng.normal(size=(N, K)) * 2.0
    return h, W, idx.astype(np.int32), logit, T


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("V,K,T", [(11, 3, 1.0), (64, 8, 2.0), (7, 7, 0.5)])
def test_uniform_teacher_and_student_closed_form(V, K, T):
    # h = 0 -> every student logit is 0 -> q = 1/V; equal teacher logits -> p = 1/K.
    # KL(p || q) over K distinct entries = sum_k (1/K) ln((1/K) / (1/V)) = ln(V/K).
    N, d = 5, 4
    rng = np.random.default_rng(1)
    h = np.zeros((N, d))
    W = rng.normal(size=(V, d))
    idx = np.stack([rng.permutation(V)[:K] for _ in range(N)]).astype(np.int32)
    logit = np.full((N, K), 3.25)
    r = oracle.fwd_bwd(h, W, idx, logit, None, T)
    assert r["loss"] == pytest.approx(math.log(V / K), rel=1e-14, abs=1e-14)
    # grad_W = G^T h = 0 because h = 0
    assert np.abs(r["grad_W"]).max() == 0.0
    # lse of an all-zero row is ln V
    assert np.allclose(r["lse"], math.log(V), rtol=1e-14)


def test_row_constant_student_gives_entropy_plus_log_v():
    # z constant along the vocabulary -> log q = -ln V for every entry, so
    # loss_r = sum_k p_k ln p_k + ln V (negative teacher entropy + ln V).
    N, d, V, K = 4, 3, 9, 4
    rng = np.random.default_rng(2)
    W = np.zeros((V, d))
    W[:, 0] = 1.0            # every vocab row equal -> z_rv = h_r0 for all v
    h = rng.normal(size=(N, d))
    idx = np.stack([rng.permutation(V)[:K] for _ in range(N)]).astype(np.int32)
    logit = rng.normal(size=(N, K))
    r = oracle.fwd_bwd(h, W, idx, logit, None, 1.0)
    for i in range(N):
        e = np.exp(logit[i] - logit[i].max())
        p = e / e.sum()
        want = float((p * np.log(p)).sum() + math.log(V))
        assert r["loss_rows"][i] == pytest.approx(want, rel=1e-13)


def test_zero_when_teacher_equals_student_full_vocab():
    # K = V, idx a permutation and teacher logits equal to the student logits:
    # p = q exactly, so the KL and both gradients vanish.  W = I makes z = h.
    V = d = 16
    N = 5
    rng = np.random.default_rng(3)
    h = np.round(rng.normal(size=(N, d)) * 8) / 8
    W = np.eye(V)
    idx = np.stack([rng.permutation(V) for _ in range(N)]).astype(np.int32)
    logit = np.take_along_axis(h, idx.astype(np.int64), axis=1)
    for T in (1.0, 2.0):
        r = oracle.fwd_bwd(h, W, idx, logit, None, T)
        assert abs(r["loss"]) < 1e-14
        assert np.abs(r["grad_h"]).max() < 1e-15
        assert np.abs(r["grad_W"]).max() < 1e-15


def test_gibbs_inequality_bound():
    # For distinct indices: sum_k p_k ln(p_k/q_k) >= -ln sum_k q_k >= 0 (log-sum inequality).
    h, W, idx, logit, T = rand_problem(N=20, d=6, V=30, K=5, seed=4)
    r = oracle.fwd_bwd(h, W, idx, logit, None, T)
    z = torch.tensor(h) @ torch.tensor(W).T
    logq = torch.log_softmax(z / T, dim=1).numpy()
    qsum = np.exp(np.take_along_axis(logq, idx.astype(np.int64), axis=1)).sum(axis=1)
    bound = -np.log(qsum)
    assert np.all(r["loss_rows"] >= bound - 1e-12)
    assert np.all(bound >= 0)


# ------------------------------------------------------------ library routines

def test_single_entry_is_cross_entropy():
    # K = 1 -> p = 1 on one index -> loss = cross-entropy of softmax(z/T) at idx.
    N, d, V, T = 7, 5, 13, 1.7
    rng = np.random.default_rng(5)
    h = rng.normal(size=(N, d))
    W = rng.normal(size=(V, d))
    tgt = rng.integers(0, V, size=N)
    r = oracle.fwd_bwd(h, W, tgt[:, None].astype(np.int32), rng.normal(size=(N, 1)), None, T)
    th = torch.tensor(h, requires_grad=True)
    tW = torch.tensor(W, requires_grad=True)
    ce = F.cross_entropy((th @ tW.T) / T, torch.tensor(tgt), reduction="mean")
    ce.backward()
    assert r["loss"] == pytest.approx(ce.item(), rel=1e-13)
    np.testing.assert_allclose(r["grad_h"], th.grad.numpy(), rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(r["grad_W"], tW.grad.numpy(), rtol=1e-11, atol=1e-14)


def test_full_vocab_teacher_is_kl_div_batchmean():
    # K = V with idx a permutation -> the top-K loss is the full KL, which
    # torch's kl_div(log q, p, reduction='batchmean') computes.
    N, d, V, T = 6, 4, 10, 2.0
    rng = np.random.default_rng(6)
    h = rng.normal(size=(N, d))
    W = rng.normal(size=(V, d))
    idx = np.stack([rng.permutation(V) for _ in range(N)]).astype(np.int32)
    logit = rng.normal(size=(N, V)) * 3
    dense_t = np.zeros((N, V))
    np.put_along_axis(dense_t, idx.astype(np.int64), logit, axis=1)
    r = oracle.fwd_bwd(h, W, idx, logit, None, T)
    th = torch.tensor(h, requires_grad=True)
    tW = torch.tensor(W, requires_grad=True)
    logq = torch.log_softmax((th @ tW.T) / T, dim=1)
    p = torch.softmax(torch.tensor(dense_t) / T, dim=1)
    kl = F.kl_div(logq, p, reduction="batchmean")
    kl.backward()
    assert r["loss"] == pytest.approx(kl.item(), rel=1e-12)
    np.testing.assert_allclose(r["grad_h"], th.grad.numpy(), rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(r["grad_W"], tW.grad.numpy(), rtol=1e-10, atol=1e-14)


def torch_dense_loss(th, tW, idx, logit, mask, T):
    """The loss written with torch primitives, differentiated by autograd."""
    logq = torch.log_softmax((th @ tW.T) / T, dim=1)
    p = torch.softmax(torch.tensor(logit) / T, dim=1)
    lq = torch.gather(logq, 1, torch.tensor(idx, dtype=torch.int64))
    per_row = (p * (torch.log(p) - lq)).sum(dim=1)
    m = torch.ones(th.shape[0], dtype=torch.bool) if mask is None else torch.tensor(mask != 0)
    return per_row[m].sum() / m.sum()


@pytest.mark.parametrize("T", [1.0, 2.0])
def test_autograd_matches(T):
    h, W, idx, logit, _ = rand_problem(N=9, d=6, V=25, K=4, seed=7)
    mask = np.array([1, 1, 0, 1, 1, 1, 0, 1, 1], np.uint8)
    r = oracle.fwd_bwd(h, W, idx, logit, mask, T)
    th = torch.tensor(h, requires_grad=True)
    tW = torch.tensor(W, requires_grad=True)
    loss = torch_dense_loss(th, tW, idx, logit, mask, T)
    loss.backward()
    assert r["loss"] == pytest.approx(loss.item(), rel=1e-13)
    np.testing.assert_allclose(r["grad_h"], th.grad.numpy(), rtol=1e-10, atol=1e-15)
    np.testing.assert_allclose(r["grad_W"], tW.grad.numpy(), rtol=1e-10, atol=1e-15)


@pytest.mark.parametrize("distinct", [True, False])
def test_grad_logits_is_autograd_in_the_logits(distinct):
    # dL/dz from autograd of the loss written on z directly (a duplicate index
    # is gathered twice, so autograd adds both probabilities)
    h, W, idx, logit, _ = rand_problem(N=10, d=6, V=21, K=5, seed=31, distinct=distinct)
    mask = np.array([1, 0, 1, 1, 1, 1, 0, 1, 1, 1], np.uint8)
    T = 1.7
    z = torch.tensor(h @ W.T, requires_grad=True)
    logq = torch.log_softmax(z / T, dim=1)
    p = torch.softmax(torch.tensor(logit) / T, dim=1)
    lq = torch.gather(logq, 1, torch.tensor(idx, dtype=torch.int64))
    per_row = (p * (torch.log(p) - lq)).sum(dim=1)
    m = torch.tensor(mask != 0)
    (per_row[m].sum() / m.sum()).backward()
    g = oracle.grad_logits(h, W, idx, logit, mask, T, block_rows=3)
    np.testing.assert_allclose(g["G"], z.grad.numpy(), rtol=1e-10, atol=1e-16)
    assert g["n_valid"] == 8 and np.all(g["G"][mask == 0] == 0)
    # and it is the factor the weight gradients are built from
    r = oracle.fwd_bwd(h, W, idx, logit, mask, T)
    np.testing.assert_allclose(g["G"] @ W, r["grad_h"], rtol=1e-12, atol=1e-16)
    np.testing.assert_allclose(g["lse"][mask != 0], r["lse"][mask != 0], rtol=1e-14)


def test_teacher_plogp_closed_forms():
    K = 6
    p = np.array([[1.0 / K] * K, [1.0, 0, 0, 0, 0, 0], [0.5, 0.5, 0, 0, 0, 0]])
    np.testing.assert_allclose(oracle.teacher_plogp(p), [-math.log(K), 0.0, -math.log(2.0)],
                               rtol=1e-15, atol=1e-16)


# ------------------------------------------------------------ finite differences

@pytest.mark.parametrize("distinct", [True, False])
def test_central_finite_differences(distinct):
    # T = 2 and a masked row so that a missing 1/T or 1/N_valid shows up; the
    # non-distinct case exercises the scatter-add of duplicate indices.
    h, W, idx, logit, _ = rand_problem(N=5, d=4, V=9, K=4, seed=8, distinct=distinct)
    T = 2.0
    mask = np.array([1, 0, 1, 1, 1], np.uint8)
    r = oracle.fwd_bwd(h, W, idx, logit, mask, T)
    eps = 1e-6

    def L(hh, WW):
        return oracle.fwd(hh, WW, idx, logit, mask, T)["loss"]

    rng = np.random.default_rng(9)
    for _ in range(12):
        i, j = rng.integers(0, h.shape[0]), rng.integers(0, h.shape[1])
        hp, hm = h.copy(), h.copy()
        hp[i, j] += eps
        hm[i, j] -= eps
        fd = (L(hp, W) - L(hm, W)) / (2 * eps)
        assert fd == pytest.approx(r["grad_h"][i, j], rel=1e-6, abs=1e-9)
        v, j = rng.integers(0, W.shape[0]), rng.integers(0, W.shape[1])
        Wp, Wm = W.copy(), W.copy()
        Wp[v, j] += eps
        Wm[v, j] -= eps
        fd = (L(h, Wp) - L(h, Wm)) / (2 * eps)
        assert fd == pytest.approx(r["grad_W"][v, j], rel=1e-6, abs=1e-9)
    # masked row: no gradient at all
    assert np.all(r["grad_h"][1] == 0.0)


# ------------------------------------------------------------ invariances

def test_temperature_identity():
    # s = (h W^T)/T and p = softmax(l/T): loss_T(h, l) = loss_1(h/T, l/T),
    # grad_h,T = grad_h,1(h/T, l/T) / T and grad_W,T = grad_W,1(h/T, l/T).
    h, W, idx, logit, _ = rand_problem(N=8, d=5, V=21, K=5, seed=10)
    T = 2.0
    a = oracle.fwd_bwd(h, W, idx, logit, None, T)
    b = oracle.fwd_bwd(h / T, W, idx, logit / T, None, 1.0)
    assert a["loss"] == pytest.approx(b["loss"], rel=1e-14)
    np.testing.assert_allclose(a["grad_h"], b["grad_h"] / T, rtol=1e-12, atol=1e-16)
    np.testing.assert_allclose(a["grad_W"], b["grad_W"], rtol=1e-12, atol=1e-16)


def test_row_block_size_invariance():
    h, W, idx, logit, T = rand_problem(N=37, d=6, V=40, K=6, seed=11)
    a = oracle.fwd_bwd(h, W, idx, logit, None, T, block_rows=256)
    b = oracle.fwd_bwd(h, W, idx, logit, None, T, block_rows=5)
    assert a["loss"] == pytest.approx(b["loss"], rel=1e-13)
    np.testing.assert_allclose(a["grad_h"], b["grad_h"], rtol=1e-12, atol=1e-16)
    np.testing.assert_allclose(a["grad_W"], b["grad_W"], rtol=1e-12, atol=1e-16)


def test_masking_a_row_equals_deleting_it_and_ignores_its_data():
    h, W, idx, logit, T = rand_problem(N=10, d=5, V=17, K=4, seed=12)
    mask = np.ones(10, np.uint8)
    mask[[2, 7]] = 0
    h2, l2 = h.copy(), logit.copy()
    h2[2] = np.nan
    l2[7] = np.nan
    a = oracle.fwd_bwd(h2, W, idx, l2, mask, T)
    keep = mask.astype(bool)
    b = oracle.fwd_bwd(h[keep], W, idx[keep], logit[keep], None, T)
    assert a["loss"] == pytest.approx(b["loss"], rel=1e-14)
    np.testing.assert_allclose(a["grad_h"][keep], b["grad_h"], rtol=1e-13)
    assert np.all(a["grad_h"][~keep] == 0)
    np.testing.assert_allclose(a["grad_W"], b["grad_W"], rtol=1e-12, atol=1e-17)


def test_permutations_and_teacher_shift():
    h, W, idx, logit, T = rand_problem(N=8, d=5, V=19, K=5, seed=13)
    a = oracle.fwd_bwd(h, W, idx, logit, None, T)
    rng = np.random.default_rng(14)
    perm_k = rng.permutation(5)
    b = oracle.fwd_bwd(h, W, idx[:, perm_k], logit[:, perm_k], None, T)
    assert a["loss"] == pytest.approx(b["loss"], rel=1e-14)
    np.testing.assert_allclose(a["grad_W"], b["grad_W"], rtol=1e-13, atol=1e-17)
    perm_n = rng.permutation(8)
    c = oracle.fwd_bwd(h[perm_n], W, idx[perm_n], logit[perm_n], None, T)
    assert a["loss"] == pytest.approx(c["loss"], rel=1e-13)
    np.testing.assert_allclose(a["grad_h"][perm_n], c["grad_h"], rtol=1e-13)
    e = oracle.fwd_bwd(h, W, idx, logit + rng.normal(size=(8, 1)) * 5, None, T)
    assert a["loss"] == pytest.approx(e["loss"], rel=1e-12)
    np.testing.assert_allclose(a["grad_h"], e["grad_h"], rtol=1e-11, atol=1e-17)


def test_gradient_sum_rule():
    # sum_v dL/dz_rv = 0 for each row (softmax sums to 1, p sums to 1), so the
    # column sums of grad_W vanish.
    h, W, idx, logit, T = rand_problem(N=12, d=6, V=33, K=7, seed=15)
    r = oracle.fwd_bwd(h, W, idx, logit, None, T)
    assert np.abs(r["grad_W"].sum(axis=0)).max() < 1e-15


# ------------------------------------------------------------ edge-case readings

def test_out_of_range_index_is_dropped_and_flagged():
    h, W, idx, logit, T = rand_problem(N=4, d=3, V=12, K=4, seed=16)
    bad = idx.copy()
    bad[1, 2] = 12
    bad[3, 0] = -1
    a = oracle.fwd_bwd(h, W, bad, logit, None, T)
    assert a["flags"] & oracle.FLAG_INDEX_RANGE
    l2 = logit.copy()
    l2[1, 2] = -np.inf
    l2[3, 0] = -np.inf
    b = oracle.fwd_bwd(h, W, idx, l2, None, T)
    assert b["flags"] == 0
    assert a["loss"] == pytest.approx(b["loss"], rel=1e-14)
    np.testing.assert_allclose(a["grad_W"], b["grad_W"], rtol=1e-13, atol=1e-17)


def test_bad_teacher_row_is_excluded_and_flagged():
    h, W, idx, logit, T = rand_problem(N=6, d=3, V=12, K=4, seed=17)
    l2 = logit.copy()
    l2[1, 3] = np.nan
    l2[4, :] = -np.inf
    a = oracle.fwd_bwd(h, W, idx, l2, None, T)
    assert a["flags"] & oracle.FLAG_BAD_TEACHER
    mask = np.array([1, 0, 1, 1, 0, 1], np.uint8)
    b = oracle.fwd_bwd(h, W, idx, logit, mask, T)
    assert a["n_valid"] == 4
    assert a["loss"] == pytest.approx(b["loss"], rel=1e-14)
    np.testing.assert_allclose(a["grad_h"], b["grad_h"], rtol=1e-13, atol=1e-17)
    np.testing.assert_allclose(a["grad_W"], b["grad_W"], rtol=1e-13, atol=1e-17)


def test_no_valid_rows_gives_zero():
    h, W, idx, logit, T = rand_problem(N=3, d=3, V=8, K=2, seed=18)
    r = oracle.fwd_bwd(h, W, idx, logit, np.zeros(3, np.uint8), T)
    assert r["loss"] == 0.0 and r["n_valid"] == 0
    assert np.all(r["grad_h"] == 0) and np.all(r["grad_W"] == 0)


def test_token_shards_with_the_batch_divisor_add_up_to_the_batch():
    # A batch split into token shards: each shard divides by the batch's
    # N_valid, so the shards' losses and grad_W add up to the batch's and
    # their grad_h rows are the batch's rows (linearity of the sum over
    # tokens); the default divisor is the shard's own count.
    h, W, idx, logit, T = rand_problem(N=9, d=4, V=13, K=3, T=2.0, seed=23)
    mask = np.array([1, 0, 1, 1, 1, 0, 1, 1, 1], np.uint8)
    full = oracle.fwd_bwd(h, W, idx, logit, mask, T)
    parts = [slice(0, 2), slice(2, 7), slice(7, 9)]
    outs = [oracle.fwd_bwd(h[s], W, idx[s], logit[s], mask[s], T, n_norm=full["n_valid"])
            for s in parts]
    assert sum(o["loss"] for o in outs) == pytest.approx(full["loss"], rel=1e-13)
    np.testing.assert_allclose(sum(o["grad_W"] for o in outs), full["grad_W"], rtol=1e-12,
                               atol=1e-16)
    np.testing.assert_allclose(np.concatenate([o["grad_h"] for o in outs]), full["grad_h"],
                               rtol=1e-12, atol=1e-16)
    own = oracle.fwd_bwd(h[2:7], W, idx[2:7], logit[2:7], mask[2:7], T)
    same = oracle.fwd_bwd(h[2:7], W, idx[2:7], logit[2:7], mask[2:7], T, n_norm=own["n_valid"])
    assert own["loss"] == same["loss"]
    assert np.array_equal(own["grad_W"], same["grad_W"])
    zero = oracle.fwd(h[:2], W, idx[:2], logit[:2], np.zeros(2, np.uint8), T, n_norm=0)
    assert zero["loss"] == 0.0


def test_minus_inf_teacher_entry_has_zero_probability():
    h, W, idx, logit, T = rand_problem(N=3, d=3, V=8, K=3, seed=19)
    l2 = logit.copy()
    l2[0, 1] = -np.inf
    a = oracle.fwd_bwd(h, W, idx, l2, None, T)
    b = oracle.fwd_bwd(h[:1], W, idx[:1, [0, 2]], logit[:1, [0, 2]], None, T)
    assert a["flags"] == 0
    assert a["loss_rows"][0] == pytest.approx(b["loss_rows"][0], rel=1e-14)


def test_sampled_rows_agree_with_dense():
    x = synth.make_inputs(40, 16, 50, 6, T=2.0, dtype="bf16", seed=20, mask="random0.2")
    a = oracle.fwd_bwd(x.h_f32(), x.W_f32(), x.idx, x.logit, x.mask, x.T)
    rows = np.array([0, 3, 17, 39])
    s = oracle.sampled_rows(x.h_f32(), x.W_f32(), x.idx, x.logit, x.mask, x.T, rows)
    assert s["n_valid"] == a["n_valid"]
    np.testing.assert_allclose(s["loss_rows"], a["loss_rows"][rows], rtol=1e-13)
    np.testing.assert_allclose(s["grad_h"], a["grad_h"][rows], rtol=1e-12, atol=1e-18)


def test_grad_W_rows_agree_with_dense():
    x = synth.make_inputs(50, 12, 60, 5, T=1.5, dtype="bf16", seed=21, mask="random0.2")
    x.idx[3, 1] = x.idx[3, 0]          # a duplicate
    a = oracle.fwd_bwd(x.h_f32(), x.W_f32(), x.idx, x.logit, x.mask, x.T)
    vr = np.array([0, 7, int(x.idx[0, 0]), int(x.idx[3, 0]), 59])
    g = oracle.grad_W_rows(x.h_f32(), x.W_f32(), x.idx, x.logit, x.mask, x.T, vr, a["lse"])
    np.testing.assert_allclose(g, a["grad_W"][vr], rtol=1e-12, atol=1e-18)


# ------------------------------------------------------------ golden regression

def test_golden_tiny_config():
    """tests/golden/config1_tiny_fp32.json was written by
    tests/golden/make_golden.py (which calls only the oracle and the input
    generator) after the pins above passed; a change in the oracle's arithmetic
    shows up here."""
    with open(os.path.join(HERE, "golden", "config1_tiny_fp32.json")) as f:
        g = json.load(f)
    x = synth.make_config(1)
    r = oracle.fwd_bwd(x.h_f32(), x.W_f32(), x.idx, x.logit, x.mask, x.T)
    assert r["loss"] == pytest.approx(g["loss"], rel=1e-12)
    assert float(np.abs(r["grad_h"]).sum()) == pytest.approx(g["grad_h_abs_sum"], rel=1e-11)
    assert float(np.abs(r["grad_W"]).sum()) == pytest.approx(g["grad_W_abs_sum"], rel=1e-11)
    np.testing.assert_allclose(r["lse"][:8], g["lse_first8"], rtol=1e-12)


def test_synth_recipe_properties():
    x = synth.make_config(1)
    assert x.h.dtype == np.float32 and x.h.shape == (64, 64)
    assert all(len(set(row)) == 8 for row in x.idx.tolist())
    assert np.all(np.diff(x.logit, axis=1) <= 0)
    y = synth.make_inputs(64, 16, 40, 5, dtype="bf16", seed=3, heavy_head=True)
    assert y.h.dtype == np.uint16
    # bf16 round trip is exact and matches round-to-nearest-even
    v = np.array([1.0, 1.00390625, 1.005859375, -2.5e-3], np.float32)
    np.testing.assert_array_equal(synth.bf16_bits_to_f32(synth.bf16_bits(v)),
                                  np.array([1.0, 1.0, 1.0078125, -0.00250244140625], np.float32))
