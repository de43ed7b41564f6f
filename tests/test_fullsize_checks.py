"""The whole-matrix checks that the full-size GPU tests apply to grad_W and
grad_h (tests/test_gpu_fullsize.py), run here on the CPU against the fp64
oracle: they must pass on exact results and on results built the way the
bf16 GPU path builds them (dL/dz = alpha g' with g' rounded to bf16, the
gradient products taking g' and bf16(alpha h)), and they must fail on planted
mistakes (the teacher term of dL/dz left out; one 256-row tile of grad_W, or
one 128-row tile of grad_h, missing)."""
import numpy as np
import pytest

import oracle
from top_kl_loss_token_b300 import synth
from test_gpu_fullsize import check_projection_identity, check_sum_rule, scaled_rows


def _bf16(a):
    return synth.bf16_bits_to_f32(synth.bf16_bits(np.asarray(a, np.float32))).astype(np.float64)


@pytest.fixture(scope="module")
def problem():
    x = synth.make_inputs(2048, 64, 3000, 16, T=2.0, dtype="bf16", seed=31, mask="random0.1")
    g = oracle.grad_logits(x.h_f32(), x.W_f32(), x.idx, x.logit, x.mask, x.T)
    G = g["G"]
    tn = x.T * g["n_valid"]
    # dL/dz as the GPU stores it: the softmax rounded to bf16 (the stored
    # exponential), then the tile G rounded to bf16
    q = np.where(g["valid"][:, None], np.exp(
        (x.h_f32().astype(np.float64) @ x.W_f32().astype(np.float64).T) / x.T
        - g["lse"][:, None]), 0.0)
    q = np.nan_to_num(q)
    Gq = _bf16(_bf16(q) / tn + (G - q / tn))
    return x, g, G, Gq


def _outputs(x, G, n_valid):
    h = x.h_f32().astype(np.float64)
    W = x.W_f32().astype(np.float64)
    valid = np.ones(x.N, bool) if x.mask is None else x.mask != 0
    return dict(grad_W=G.T @ np.where(valid[:, None], h, 0.0), grad_h=G @ W, n_valid=n_valid)


def _scaled_outputs(x, G, n_valid, seed=3):
    """The bf16 path's products: per valid row a factor alpha (here random,
    of the size 1 / (T N_valid) times a power-of-two spread), g' = bf16(G /
    alpha), grad_h = alpha (g' W), grad_W = g'^T bf16(alpha h)."""
    rng = np.random.default_rng(seed)
    W = x.W_f32().astype(np.float64)
    valid = np.ones(x.N, bool) if x.mask is None else x.mask != 0
    rows = np.nonzero(valid)[0]
    alpha = (2.0 ** rng.uniform(-6, 6, size=rows.size) / (x.T * n_valid)).astype(np.float32)
    alpha = alpha.astype(np.float64)
    gp = _bf16(G[rows] / alpha[:, None])
    grad_h = np.zeros((x.N, x.d))
    grad_h[rows] = alpha[:, None] * (gp @ W)
    grad_W = gp.T @ scaled_rows(x, rows, alpha)
    return dict(grad_W=grad_W, grad_h=grad_h, n_valid=n_valid, rows=rows), alpha


def test_checks_pass_on_exact_and_on_rounded_results(problem):
    x, g, G, Gq = problem
    exact = _outputs(x, G, g["n_valid"])
    assert check_sum_rule(x, exact) < 0.05
    assert check_projection_identity(x, exact) < 1e-12
    rounded = _outputs(x, Gq, g["n_valid"])
    assert check_sum_rule(x, rounded) <= 1.0
    check_projection_identity(x, rounded)
    scaled, alpha = _scaled_outputs(x, Gq, g["n_valid"])
    assert check_sum_rule(x, scaled) <= 1.0
    assert check_projection_identity(x, scaled, alpha) < 1e-10
    # without the factors the identity is off by the rounding of alpha h
    with pytest.raises(AssertionError):
        check_projection_identity(x, dict(scaled, grad_h=scaled["grad_h"] * 1.01), alpha)


def test_sum_rule_catches_a_missing_teacher_term(problem):
    x, g, G, Gq = problem
    # dL/dz without the teacher's subtraction: the softmax term alone
    valid = np.ones(x.N, bool) if x.mask is None else x.mask != 0
    p_scat = np.zeros_like(G)
    r = np.repeat(np.arange(x.N), x.K)
    np.add.at(p_scat, (r, x.idx.reshape(-1).astype(np.int64)), g["p"].reshape(-1))
    no_teacher = G + p_scat / (x.T * g["n_valid"]) * valid[:, None]
    with pytest.raises(AssertionError):
        check_sum_rule(x, _outputs(x, no_teacher, g["n_valid"]))


@pytest.mark.parametrize("scaled", [False, True])
def test_projection_identity_catches_a_missing_tile(problem, scaled):
    x, g, G, Gq = problem
    if scaled:
        out, alpha = _scaled_outputs(x, Gq, g["n_valid"])
    else:
        out, alpha = _outputs(x, Gq, g["n_valid"]), None
    bad = dict(out)
    bad["grad_W"] = out["grad_W"].copy()
    bad["grad_W"][512:768] = 0.0
    with pytest.raises(AssertionError):
        check_projection_identity(x, bad, alpha)
    bad = dict(out)
    bad["grad_h"] = out["grad_h"].copy()
    bad["grad_h"][1024:1152] = 0.0
    with pytest.raises(AssertionError):
        check_projection_identity(x, bad, alpha)


# ------------------------------------------------- the full-vocabulary loss

@pytest.fixture(scope="module")
def full_problem():
    xs, xt = synth.make_full_teacher_pair(2, N=2048, d=64, V=3000, T=2.0, mask="random0.1",
                                          seed=41)
    g = oracle.full_kl_grad_logits(xs.h_f32(), xs.W_f32(), xt.h_f32(), xt.W_f32(), xs.mask,
                                   xs.T)
    tn = xs.T * g["n_valid"]
    # the tile as the GPU builds it: both stored exponentials rounded to bf16
    # (a power-of-two block reference does not change their rounding), the
    # per-block factors applied, the difference rounded to bf16 once more
    Gq = _bf16((_bf16(g["q"]) - _bf16(g["p"])) / tn)
    return xs, g, Gq


def test_full_vocabulary_checks_pass_on_rounded_results(full_problem):
    xs, g, Gq = full_problem
    exact = _outputs(xs, g["G"], g["n_valid"])
    assert check_sum_rule(xs, exact, rounding=4.01) < 0.05
    assert check_projection_identity(xs, exact) < 1e-12
    rounded = _outputs(xs, Gq, g["n_valid"])
    assert check_sum_rule(xs, rounded, rounding=4.01) <= 1.0
    check_projection_identity(xs, rounded)


def test_full_vocabulary_checks_catch_planted_mistakes(full_problem):
    xs, g, Gq = full_problem
    tn = xs.T * g["n_valid"]
    # the teacher's distribution left out of dL/dz_s
    with pytest.raises(AssertionError):
        check_sum_rule(xs, _outputs(xs, _bf16(g["q"] / tn), g["n_valid"]), rounding=4.01)
    # the teacher term without its temperature
    with pytest.raises(AssertionError):
        check_sum_rule(xs, _outputs(xs, _bf16(g["q"] / tn - g["p"] / g["n_valid"]),
                                    g["n_valid"]), rounding=4.01)
    out = _outputs(xs, Gq, g["n_valid"])
    bad = dict(out)
    bad["grad_W"] = out["grad_W"].copy()
    bad["grad_W"][512:768] = 0.0
    with pytest.raises(AssertionError):
        check_projection_identity(xs, bad)
