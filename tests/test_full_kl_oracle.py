"""Pins of the fp64 full-vocabulary (K = V) loss oracle
(oracle/full_kl_oracle.py) to things other than itself: torch's KL divergence
(batchmean) and its autograd through the two matrix products, zero at
teacher = student, Gibbs' inequality, central finite differences, mask =
deletion, the empty batch, and agreement with the separately written top-K
oracle when the cache holds the whole vocabulary.  Planted mistakes at the
end must each fail one of them."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import full_kl_oracle as fko


def _inputs(seed, N=12, ds=8, dt=6, V=40, scale=0.7):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((N, ds)) * scale, rng.standard_normal((V, ds)) * scale,
            rng.standard_normal((N, dt)) * scale, rng.standard_normal((V, dt)) * scale)


def _torch_loss(hs, Ws, ht, Wt, T, rows):
    s = (hs[rows] @ Ws.T) / T
    t = (ht[rows] @ Wt.T) / T
    return F.kl_div(F.log_softmax(s, dim=1), F.softmax(t, dim=1), reduction="batchmean")


@pytest.mark.parametrize("T", [1.0, 2.0])
def test_kl_div_batchmean_and_its_autograd(T):
    hs, Ws, ht, Wt = _inputs(1)
    mask = np.ones(12, np.uint8)
    mask[[2, 7]] = 0
    r = fko.full_kl_fwd_bwd(hs, Ws, ht, Wt, mask, T, block_rows=5)
    rows = torch.from_numpy(np.nonzero(mask)[0])
    ths = torch.tensor(hs, requires_grad=True)
    tWs = torch.tensor(Ws, requires_grad=True)
    loss = _torch_loss(ths, tWs, torch.tensor(ht), torch.tensor(Wt), T, rows)
    loss.backward()
    assert r["loss"] == pytest.approx(loss.item(), rel=1e-12)
    np.testing.assert_allclose(r["grad_h"], ths.grad.numpy(), rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(r["grad_W"], tWs.grad.numpy(), rtol=1e-10, atol=1e-14)


def test_grad_logits_is_autograd_of_kl_div_in_the_student_logits():
    hs, Ws, ht, Wt = _inputs(9)
    mask = np.ones(12, np.uint8)
    mask[[0, 5]] = 0
    T = 1.5
    rows = torch.from_numpy(np.nonzero(mask)[0])
    z = torch.tensor(hs @ Ws.T, requires_grad=True)
    t = torch.tensor(ht @ Wt.T)
    F.kl_div(F.log_softmax(z[rows] / T, dim=1), F.softmax(t[rows] / T, dim=1),
             reduction="batchmean").backward()
    g = fko.full_kl_grad_logits(hs, Ws, ht, Wt, mask, T)
    np.testing.assert_allclose(g["G"], z.grad.numpy(), rtol=1e-10, atol=1e-16)
    assert g["n_valid"] == 10 and np.all(g["G"][mask == 0] == 0)
    np.testing.assert_allclose(g["q"][mask != 0].sum(axis=1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(g["p"][mask != 0].sum(axis=1), 1.0, rtol=1e-14)


def test_zero_when_student_equals_teacher():
    hs, Ws, _, _ = _inputs(2)
    r = fko.full_kl_fwd_bwd(hs, Ws, hs, Ws, None, 1.5)
    assert abs(r["loss"]) < 1e-14
    assert np.abs(r["grad_h"]).max() < 1e-14 and np.abs(r["grad_W"]).max() < 1e-14


def test_gibbs_inequality():
    for seed in range(5):
        r = fko.full_kl_fwd_bwd(*_inputs(10 + seed, scale=2.0), None, 1.0)
        assert np.all(r["loss_rows"] >= -1e-14)


def test_central_finite_differences():
    hs, Ws, ht, Wt = _inputs(3, N=5, V=17)
    T = 2.0
    r = fko.full_kl_fwd_bwd(hs, Ws, ht, Wt, None, T)
    eps = 1e-6
    for (arr, grad, idx) in ((hs, r["grad_h"], (1, 3)), (Ws, r["grad_W"], (4, 2)),
                             (Ws, r["grad_W"], (16, 7))):
        a = arr.copy()
        a[idx] += eps
        lp = fko.full_kl_fwd_bwd(*(a if x is arr else x for x in (hs, Ws, ht, Wt)), None, T)["loss"]
        a[idx] -= 2 * eps
        lm = fko.full_kl_fwd_bwd(*(a if x is arr else x for x in (hs, Ws, ht, Wt)), None, T)["loss"]
        assert (lp - lm) / (2 * eps) == pytest.approx(grad[idx], rel=1e-6, abs=1e-12)


def test_masked_rows_equal_deletion_and_ignore_their_data():
    hs, Ws, ht, Wt = _inputs(4)
    mask = np.ones(12, np.uint8)
    mask[[0, 5, 11]] = 0
    hs2, ht2 = hs.copy(), ht.copy()
    hs2[mask == 0] = np.nan
    ht2[mask == 0] = np.nan
    a = fko.full_kl_fwd_bwd(hs2, Ws, ht2, Wt, mask, 1.0)
    keep = mask != 0
    b = fko.full_kl_fwd_bwd(hs[keep], Ws, ht[keep], Wt, None, 1.0)
    assert a["loss"] == pytest.approx(b["loss"], rel=1e-13)
    np.testing.assert_allclose(a["grad_W"], b["grad_W"], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(a["grad_h"][keep], b["grad_h"], rtol=1e-12, atol=1e-15)
    assert np.all(a["grad_h"][~keep] == 0)


def test_empty_batch_is_zero():
    hs, Ws, ht, Wt = _inputs(5)
    r = fko.full_kl_fwd_bwd(hs, Ws, ht, Wt, np.zeros(12, np.uint8), 1.0)
    assert r["loss"] == 0.0 and r["n_valid"] == 0
    assert np.all(r["grad_h"] == 0) and np.all(r["grad_W"] == 0)


def test_equals_top_k_oracle_with_the_whole_vocabulary_cached():
    hs, Ws, ht, Wt = _inputs(6)
    T = 1.7
    mask = np.ones(12, np.uint8)
    mask[3] = 0
    r = fko.full_kl_fwd_bwd(hs, Ws, ht, Wt, mask, T)
    zt = ht @ Wt.T
    rng = np.random.default_rng(0)
    idx = np.stack([rng.permutation(40) for _ in range(12)]).astype(np.int32)
    logit = np.take_along_axis(zt, idx, axis=1)
    k = oracle.fwd_bwd(hs, Ws, idx, logit, mask, T)
    assert r["loss"] == pytest.approx(k["loss"], rel=1e-11)
    np.testing.assert_allclose(r["grad_W"], k["grad_W"], rtol=1e-9, atol=1e-14)
    np.testing.assert_allclose(r["grad_h"], k["grad_h"], rtol=1e-9, atol=1e-14)


def test_sampled_rows_match_the_full_computation():
    hs, Ws, ht, Wt = _inputs(7)
    mask = np.ones(12, np.uint8)
    mask[[1, 9]] = 0
    r = fko.full_kl_fwd_bwd(hs, Ws, ht, Wt, mask, 2.0)
    rows = np.array([0, 1, 4, 9, 11])
    s = fko.full_kl_sampled_rows(hs, Ws, ht, Wt, mask, 2.0, rows)
    np.testing.assert_allclose(s["grad_h"], r["grad_h"][rows], rtol=1e-12, atol=1e-15)
    v = s["valid"]
    np.testing.assert_allclose(s["loss_rows"], r["loss_rows"][rows], rtol=1e-12)
    assert np.all(s["loss_rows"][~v] == 0) and np.all(s["grad_h"][~v] == 0)
    np.testing.assert_allclose(s["lse_s"][v], r["lse_s"][rows][v], rtol=1e-12)


def test_sampled_grad_W_rows_are_autograd_of_kl_div():
    # the column-sampled grad_W (used at full size, where the dense one is out
    # of reach) against torch autograd of F.kl_div, and the per-row logsumexps
    # it takes against torch.logsumexp
    hs, Ws, ht, Wt = _inputs(11, N=20, V=50)
    mask = np.ones(20, np.uint8)
    mask[[3, 4, 17]] = 0
    T = 2.0
    r = fko.full_kl_fwd_bwd(hs, Ws, ht, Wt, mask, T, block_rows=7)
    v = mask != 0
    np.testing.assert_allclose(r["lse_t"][v], torch.logsumexp(torch.tensor(ht @ Wt.T) / T,
                                                              dim=1).numpy()[v], rtol=1e-13)
    np.testing.assert_allclose(r["lse_s"][v], torch.logsumexp(torch.tensor(hs @ Ws.T) / T,
                                                              dim=1).numpy()[v], rtol=1e-13)
    rows = torch.from_numpy(np.nonzero(mask)[0])
    tWs = torch.tensor(Ws, requires_grad=True)
    _torch_loss(torch.tensor(hs), tWs, torch.tensor(ht), torch.tensor(Wt), T, rows).backward()
    vr = np.array([0, 7, 8, 31, 49])
    got = fko.full_kl_grad_W_rows(hs, Ws, ht, Wt, mask, T, vr, r["lse_s"], r["lse_t"],
                                  block_rows=6)
    np.testing.assert_allclose(got, tWs.grad.numpy()[vr], rtol=1e-10, atol=1e-15)


# ------------------------------------------------------------ planted mistakes

PINS = [lambda: test_kl_div_batchmean_and_its_autograd(2.0), test_zero_when_student_equals_teacher,
        test_central_finite_differences, test_masked_rows_equal_deletion_and_ignore_their_data,
        test_gibbs_inequality]


def _mutant(kind):
    real_ls = fko._log_softmax

    def run(h_s, W_s, h_t, W_t, mask, T, block_rows=256, want_grads=True):
        h_s = np.asarray(h_s, dtype=np.float64); W_s = np.asarray(W_s, dtype=np.float64)
        h_t = np.asarray(h_t, dtype=np.float64); W_t = np.asarray(W_t, dtype=np.float64)
        N = h_s.shape[0]
        valid = np.ones(N, dtype=bool) if mask is None else np.asarray(mask) != 0
        nv = int(valid.sum())
        rows = np.nonzero(valid)[0]
        t = (h_t[rows] @ W_t.T) / (1.0 if kind == "teacher_without_T" else T)
        s = (h_s[rows] @ W_s.T) / T
        logp, logq = real_ls(t), real_ls(s)
        p = np.exp(logp)
        lr = np.zeros(N)
        lr[rows] = (p * (logp - logq)).sum(axis=1)
        if kind == "reverse_kl":
            q = np.exp(logq)
            lr[rows] = (q * (logq - logp)).sum(axis=1)
        denom = T * (N if kind == "mean_over_all_rows" else nv)
        if kind == "no_T_in_grad":
            denom = nv
        G = (np.exp(logq) - p) / denom
        if kind == "grad_sign":
            G = -G
        gh = np.zeros_like(h_s)
        gh[rows] = G @ W_s
        gW = G.T @ h_s[rows]
        loss = float(lr[valid].sum() / (N if kind == "mean_over_all_rows" else nv)) if nv else 0.0
        return dict(loss=loss, grad_h=gh, grad_W=gW, loss_rows=lr, lse_s=np.zeros(N),
                    valid=valid, n_valid=nv)
    return run


@pytest.mark.parametrize("kind", ["teacher_without_T", "reverse_kl", "mean_over_all_rows",
                                  "no_T_in_grad", "grad_sign"])
def test_planted_mistake_is_caught(kind, monkeypatch):
    monkeypatch.setattr(fko, "full_kl_fwd_bwd", _mutant(kind))
    failed = False
    for p in PINS:
        try:
            with np.errstate(all="ignore"):
                p()
        except AssertionError:
            failed = True
            break
    assert failed, kind
