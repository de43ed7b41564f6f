"""Planted mistakes in the oracle must be caught by its pins.

Each case swaps the oracle's row-block routine or teacher routine for a copy
with one plausible mistake (a dropped term, a wrong sign, a missing 1/T or
1/N_valid, a transposed operand, a wrong normalisation) and checks that at
least one of the pins in test_oracle.py fails.  Runs on the CPU only."""
import numpy as np
import pytest

import oracle
from oracle import kd_oracle as ko
import test_oracle as pins

PINS = [
    lambda: pins.test_uniform_teacher_and_student_closed_form(11, 3, 1.0),
    lambda: pins.test_uniform_teacher_and_student_closed_form(64, 8, 2.0),
    pins.test_row_constant_student_gives_entropy_plus_log_v,
    pins.test_zero_when_teacher_equals_student_full_vocab,
    pins.test_gibbs_inequality_bound,
    pins.test_single_entry_is_cross_entropy,
    pins.test_full_vocab_teacher_is_kl_div_batchmean,
    lambda: pins.test_autograd_matches(2.0),
    lambda: pins.test_central_finite_differences(True),
    lambda: pins.test_central_finite_differences(False),
    pins.test_gradient_sum_rule,
    pins.test_masking_a_row_equals_deleting_it_and_ignores_its_data,
]


def some_pin_fails():
    for p in PINS:
        try:
            with np.errstate(all="ignore"):
                p()
        except (AssertionError, ValueError, IndexError):
            return True
    return False


def _mutated_row_block(kind):
    orig = ko._row_block

    def f(H, W, idx, p, valid, T, n_valid):
        H = np.where(valid[:, None], H, 0.0)
        S = (H @ W.T) / (1.0 if kind == "no_T_in_logits" else T)
        m = S.max(axis=1, keepdims=True)
        lse = (m + np.log(np.exp(S - m).sum(axis=1, keepdims=True)))[:, 0]
        if kind == "lse_without_max":
            lse = np.log(np.exp(S - m).sum(axis=1))
        V = W.shape[0]
        in_range = (idx >= 0) & (idx < V)
        safe = np.where(in_range, idx, 0)
        s_idx = np.take_along_axis(S, safe, axis=1)
        pk = np.where(in_range, p, 0.0)
        plogp = ko._plogp(pk)
        if kind == "drop_plogp":
            plogp = 0.0 * plogp
        sign = -1.0 if kind == "wrong_sign" else 1.0
        loss_rows = plogp - sign * (pk * (s_idx - lse[:, None])).sum(axis=1)
        loss_rows = np.where(valid, loss_rows, 0.0)
        G = np.exp(S - lse[:, None])
        r = np.repeat(np.arange(H.shape[0]), idx.shape[1])
        if kind == "scatter_overwrite":
            G[r, safe.reshape(-1)] = G[r, safe.reshape(-1)] - pk.reshape(-1)
        elif kind != "drop_teacher_grad":
            np.add.at(G, (r, safe.reshape(-1)), -pk.reshape(-1))
        if kind == "no_T_in_grad":
            G /= max(n_valid, 1)
        elif kind == "no_nvalid_in_grad":
            G /= T
        elif kind == "T_squared":
            G /= (T * T * max(n_valid, 1))
        else:
            G /= (T * max(n_valid, 1))
        G[~valid] = 0.0
        return lse, loss_rows, G

    return f, orig


def _mutated_teacher(kind):
    orig = ko.teacher_distribution

    def f(topk_idx, topk_logit, mask, V, T):
        p, valid, flags = orig(topk_idx, topk_logit, mask, V, T if kind != "teacher_no_T" else 1.0)
        if kind == "teacher_unnormalised":
            lg = np.asarray(topk_logit, dtype=np.float64)
            p = np.where(valid[:, None], np.exp(lg / T - (lg / T).max()), 0.0)
        return p, valid, flags

    return f, orig


@pytest.mark.parametrize("kind", ["no_T_in_logits", "lse_without_max", "drop_plogp", "wrong_sign",
                                  "scatter_overwrite", "drop_teacher_grad", "no_T_in_grad",
                                  "no_nvalid_in_grad", "T_squared"])
def test_row_block_mutation_is_caught(monkeypatch, kind):
    f, _ = _mutated_row_block(kind)
    monkeypatch.setattr(ko, "_row_block", f)
    assert some_pin_fails(), kind


@pytest.mark.parametrize("kind", ["teacher_no_T", "teacher_unnormalised"])
def test_teacher_mutation_is_caught(monkeypatch, kind):
    f, _ = _mutated_teacher(kind)
    monkeypatch.setattr(ko, "teacher_distribution", f)
    assert some_pin_fails(), kind


def test_transposed_grad_W_is_caught(monkeypatch):
    orig = ko.fwd_bwd

    def f(*a, **k):
        r = orig(*a, **k)
        if r["grad_W"] is not None and r["grad_W"].shape[0] == r["grad_W"].shape[1]:
            r["grad_W"] = r["grad_W"].T.copy()
        return r

    monkeypatch.setattr(ko, "fwd_bwd", f)
    monkeypatch.setattr(oracle, "fwd_bwd", f)
    # the K = V zero-loss pin uses d = V (square grad_W); a transpose of a
    # random square grad_W is caught by autograd / finite differences on square shapes
    def square_autograd():
        h, W, idx, logit, _ = pins.rand_problem(N=7, d=9, V=9, K=3, seed=33)
        r = oracle.fwd_bwd(h, W, idx, logit, None, 1.0)
        import torch
        th = torch.tensor(h, requires_grad=True)
        tW = torch.tensor(W, requires_grad=True)
        pins.torch_dense_loss(th, tW, idx, logit, None, 1.0).backward()
        np.testing.assert_allclose(r["grad_W"], tW.grad.numpy(), rtol=1e-10, atol=1e-15)
    with pytest.raises(AssertionError):
        square_autograd()


def test_unmutated_oracle_passes_every_pin():
    assert not some_pin_fails()
