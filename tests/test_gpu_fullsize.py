"""Parity at the full workload sizes, in the launch configuration bench.py
times (default chunk), against the fp64 oracle:
  * the whole-batch loss, every token's lse and loss term (the oracle's full
    dense forward, computed once per input set and cached by
    tests/golden/make_fullsize_oracle.py);
  * 2048 grad_h rows (plus the edges of mask runs) and about 2048 grad_W rows
    (half at teacher indices), each computed by the oracle on its own (grad_W
    rows from the oracle's own lse);
and properties that hold at any size and cover every element:
  * the gradient sum rule: softmax and the teacher distribution both sum to
    one per token, so sum_v dL/dz_rv = 0 and every column of grad_W sums to 0
    (up to the bf16 rounding of the stored dL/dz tile, bounded below);
  * W^T grad_W = grad_h^T h (both are (dL/dz W)^T h), projected on random
    vectors: one grad_W or grad_h tile missing or misplaced breaks it;
  * the loss is the mean of the per-token terms; grad_W is additive over a
    split of the tokens; results do not depend on the chunk."""
import numpy as np
import pytest

import oracle
from top_kl_loss_token_b300 import synth
from kd_testutil import TOL, fullsize_full_oracle, fullsize_oracle, max_rel_err, run_gpu, to_device

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def sample_rows(x, n=2048, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(x.N, size=min(n, x.N), replace=False).tolist())
    rows |= {0, x.N - 1}
    if x.mask is not None:
        edges = np.nonzero(np.diff(x.mask.astype(np.int8)))[0]
        for e in edges[:16]:
            rows |= {int(e), int(e) + 1}
    return np.array(sorted(rows))


def check_sampled(kd, x, got, rows):
    ref = oracle.sampled_rows(x.h_f32(), x.W_f32(), x.idx, x.logit, x.mask, x.T, rows)
    assert got["n_valid"] == ref["n_valid"]
    tl, tg = TOL[x.dtype]
    # GPU per-row results are stored in compacted order; map original rows.
    pos = {int(r): i for i, r in enumerate(got["rows"])}
    v = ref["valid"]
    gi = np.array([pos[int(r)] for r in rows[v]])
    np.testing.assert_allclose(got["lse"][gi], ref["lse"][v], rtol=tl, atol=tl)
    # per-token loss terms at the loss tolerance (absolute floor: that
    # tolerance of the mean term, for terms near zero)
    lscale = float(np.abs(ref["loss_rows"][v]).mean())
    np.testing.assert_allclose(got["loss_rows"][gi], ref["loss_rows"][v], rtol=tl,
                               atol=tl * lscale)
    gh = got["grad_h"][rows]
    assert max_rel_err(gh, ref["grad_h"]) <= tg
    assert np.all(got["grad_h"][rows[~v]] == 0)
    # the loss is the mean of the per-token terms
    assert got["loss"] == pytest.approx(float(np.mean(got["loss_rows"].astype(np.float64))), rel=1e-6)
    return ref


def check_whole_batch(x, got, full):
    """The GPU's loss, lse and loss terms of every valid token against the
    oracle's full forward."""
    tl, _ = TOL[x.dtype]
    assert got["n_valid"] == int(full["n_valid"])
    assert abs(got["loss"] - float(full["loss"])) <= tl * abs(float(full["loss"])), \
        (got["loss"], float(full["loss"]))
    rows = got["rows"]
    lse = full["lse"][rows]
    lr = full["loss_rows"][rows]
    np.testing.assert_allclose(got["lse"], lse, rtol=tl, atol=tl)
    np.testing.assert_allclose(got["loss_rows"], lr, rtol=tl, atol=tl * float(np.abs(lr).mean()))


def check_grad_W_rows(x, got, full):
    """Sampled grad_W rows (teacher rank-1 indices, uniform rows, the first
    and the last) against the oracle; max-abs error relative to their max."""
    _, tg = TOL[x.dtype]
    vr = full["vocab_rows"]
    assert max_rel_err(got["grad_W"][vr], full["grad_W_rows"]) <= tg


def check_sum_rule(x, got, rounding=3.01):
    """Every column of grad_W sums to ~0.

    Exactly, sum_v dL/dz_rv = (sum_v q_rv - sum_k p_rk) / (T N_valid) = 0.  The
    GPU's stored tile G~ carries two bf16 roundings (the exponential u, then
    the tile): |G~ - G| <= 2^-9 (q / (T N_valid)) + 2^-9 |G|, so per token
    |sum_v G~_rv| <= e = 3.01 * 2^-9 / (T N_valid).  These per-token errors
    are zero-mean and independent across tokens, so column j's sum
    sum_r e_r h_rj stays below 8 e sqrt(sum_r h_rj^2) (Hoeffding: a chance
    of 2e-14 per column).  Added: 1e-5 of sum_r |h_rj| / (T N_valid) for the
    fp32 logsumexp and teacher sums (a per-token offset, not zero-mean) and
    1e-5 of sum_v |grad_W_vj| for the fp32 accumulation.  Dropping the
    teacher term would give |sum_r h_rj| / (T N_valid), about 20 times the
    bound.  The full-vocabulary loss stores G~ = bf16(alpha_s u~_s - alpha_t
    u~_t) with both exponentials rounded once: 2^-9 (q + p) from them and
    2^-9 (q + p) from the tile, so e = 4.01 * 2^-9 / (T N_valid) there
    (`rounding`)."""
    gW = got["grad_W"]
    h = x.h_f32().astype(np.float64)
    valid = np.ones(x.N, bool) if x.mask is None else x.mask != 0
    hv = h[valid]
    tn = x.T * got["n_valid"]
    e = rounding * 2.0 ** -9 / tn
    bound = (8.0 * e * np.sqrt((hv * hv).sum(axis=0)) + 1e-5 * np.abs(hv).sum(axis=0) / tn
             + 1e-5 * np.abs(gW).sum(axis=0))
    colsum = gW.sum(axis=0)
    worst = float(np.max(np.abs(colsum) / bound))
    assert worst <= 1.0, f"column sum {worst:.3f} x its bound"
    return worst


def scaled_rows(x, rows, alpha):
    """The chunk rows of h as the bf16 path hands them to the grad_W product:
    alpha_i h_r (fp32 product) rounded to bf16."""
    from top_kl_loss_token_b300 import synth
    hs = x.h_f32()[rows] * alpha.astype(np.float32)[:, None]
    return synth.bf16_bits_to_f32(synth.bf16_bits(hs)).astype(np.float64)


def row_factors(kd, got, N):
    """alpha_i of every valid row (compacted order) from the call's workspace."""
    import torch
    rs = kd.workspace_view(got["ws"], got["lay"], "rowstat", 4 * N, torch.float32).cpu().numpy()
    return rs[2 * N: 2 * N + got["n_valid"]].astype(np.float64)


def check_projection_identity(x, got, alpha=None, n_vec=4, seed=0):
    """(W c)^T grad_W = sum_r ((grad_h_r . c) / alpha_r) h~_r for random c.

    The bf16 path stores g' with dL/dz = alpha g' and hands the gradient
    products g' and h~ = bf16(alpha h): grad_h_r = alpha_r (g'_r W) and
    grad_W = g'^T h~.  Both sides are then c^T W^T g'^T h~ over the same
    stored operands; they differ only by the fp32 accumulation order of the
    tensor cores (relative about 2^-24 sqrt(V) < 1e-4), so 1e-3 of the
    largest entry leaves a wide margin, while a missing 256-row tile of
    grad_W, or 128-row tile of grad_h, moves the projection by about
    sqrt(256 / V), several percent.  alpha None: alpha = 1 and h~ = h
    (dL/dz stored as it is)."""
    rng = np.random.default_rng(seed)
    W = x.W_f32().astype(np.float64)
    valid = np.ones(x.N, bool) if x.mask is None else x.mask != 0
    rows = got["rows"] if "rows" in got else np.nonzero(valid)[0]
    C = rng.standard_normal((x.d, n_vec))
    if alpha is None:
        a = np.ones(len(rows))
        ht = x.h_f32().astype(np.float64)[rows]
    else:
        a = alpha
        ht = scaled_rows(x, rows, alpha)
    lhs = (W @ C).T @ got["grad_W"]
    rhs = ((got["grad_h"][rows] @ C) / a[:, None]).T @ ht
    err = float(np.abs(lhs - rhs).max() / np.abs(rhs).max())
    assert err <= 1e-3, err
    return err


@pytest.mark.parametrize("cfg", [3, 5, 4])
def test_full_size_against_the_oracle(kd, cfg):
    x = synth.make_config(cfg)
    got = run_gpu(kd, x)
    assert got["err"] == 0
    full = fullsize_oracle(cfg, x)
    check_whole_batch(x, got, full)
    check_sampled(kd, x, got, sample_rows(x, seed=cfg))
    check_grad_W_rows(x, got, full)
    check_sum_rule(x, got)
    check_projection_identity(x, got, row_factors(kd, got, x.N))


def test_full_size_llama_config_with_grad_W_rows(kd):
    x = synth.make_config(2)
    got = run_gpu(kd, x)
    assert got["err"] == 0
    full = oracle.fwd(x.h_f32(), x.W_f32(), x.idx, x.logit, x.mask, x.T, block_rows=512)
    assert abs(got["loss"] - full["loss"]) <= TOL["bf16"][0] * abs(full["loss"])
    check_sampled(kd, x, got, sample_rows(x, seed=2))
    rng = np.random.default_rng(22)
    vr = np.unique(np.concatenate([x.idx[rng.integers(0, x.N, 1024), 0],
                                   rng.integers(0, x.V, 1024), [0, x.V - 1]]))
    ref = oracle.grad_W_rows(x.h_f32(), x.W_f32(), x.idx, x.logit, x.mask, x.T, vr, full["lse"])
    # max-abs error against max|grad_W| over the sampled rows
    assert max_rel_err(got["grad_W"][vr], ref) <= TOL["bf16"][1]
    check_sum_rule(x, got)
    check_projection_identity(x, got, row_factors(kd, got, x.N))


def test_full_size_chunk_invariance_and_token_split(kd):
    import torch
    x = synth.make_config(3)
    t = to_device(x)
    a = run_gpu(kd, x, tensors=t)
    b = run_gpu(kd, x, chunk=16384, tensors=t)
    assert abs(a["loss"] - b["loss"]) <= 1e-5 * abs(a["loss"])
    assert max_rel_err(b["grad_h"], a["grad_h"]) <= 2e-3
    assert max_rel_err(b["grad_W"], a["grad_W"]) <= 2e-3
    # grad_W is a sum over tokens: N * grad_W(all) = N1 * grad_W(first half) + N2 * grad_W(second half)
    N = x.N
    m1 = np.zeros(N, np.uint8)
    m1[: N // 3] = 1
    h, W, idx, lg, _ = t
    x1 = synth.KDInputs(x.name, x.dtype, x.h, x.W, x.idx, x.logit, m1, x.T, x.seed)
    x2 = synth.KDInputs(x.name, x.dtype, x.h, x.W, x.idx, x.logit, 1 - m1, x.T, x.seed)
    g1 = run_gpu(kd, x1, tensors=(h, W, idx, lg, torch.from_numpy(m1).cuda()))
    g2 = run_gpu(kd, x2, tensors=(h, W, idx, lg, torch.from_numpy(1 - m1).cuda()))
    comb = (g1["grad_W"] * g1["n_valid"] + g2["grad_W"] * g2["n_valid"]) / N
    # Unlike the chunk change above, the split changes N_valid, so each run
    # scales its bf16 gradient tile by a different 1/(T N_valid) and rounds it
    # on its own: the stored exponentials (rel. up to 2^-8 on q, bf16 has an
    # 8-bit significand) and the tile itself (up to 2^-8 on G) carry up to
    # 2^-8 (|q| + |G|), and the two runs' roundings are independent: allow
    # 2^-7 = 7.8e-3 of the largest entry.
    assert max_rel_err(comb, a["grad_W"]) <= 4 * 2.0 ** -9
    lcomb = (g1["loss"] * g1["n_valid"] + g2["loss"] * g2["n_valid"]) / N
    assert lcomb == pytest.approx(a["loss"], rel=1e-5)


def test_full_size_forward_only_matches_fwd_bwd(kd):
    # kd_topk_kl_fwd runs the same teacher preparation, pass 1 and logsumexp
    # kernels without the gradient part.  Its blocks sum their exponentials
    # relative to their own maxima, the bf16 fwd+bwd relative to one reference
    # per row: the same lse and loss up to fp32 rounding.
    x = synth.make_config(3)
    t = to_device(x)
    a = run_gpu(kd, x, tensors=t)
    b = run_gpu(kd, x, tensors=t, want_grads=False)
    assert a["err"] == 0 and b["err"] == 0
    assert b["loss"] == pytest.approx(a["loss"], rel=1e-6)
    np.testing.assert_array_equal(b["rows"], a["rows"])
    np.testing.assert_allclose(b["lse"], a["lse"], rtol=1e-6)


def test_full_vocabulary_loss_at_full_size(kd):
    """The full-vocabulary loss (kd_full_kl_fwd_bwd) on config 3's sizes in
    the launch configuration `bench.py --full-teacher` times: 32K tokens,
    d_s = d_t = 2880, V = 201,088, the default 4096-token chunk (8 chunks,
    grad_W accumulated over them).  Against the full-vocabulary oracle: the
    whole-batch loss, every token's lse and loss term, sampled grad_h and
    grad_W rows; the sum rule and the projection identity on all of grad_W."""
    import torch
    xs, xt = synth.make_full_teacher_pair(3)
    full = fullsize_full_oracle(3, xs, xt)
    hs, Ws, _, _, mask = to_device(xs)
    ht, Wt = to_device(xt)[:2]
    N, d, V = xs.N, xs.d, xs.V
    err = torch.zeros(1, dtype=torch.int32, device=hs.device)
    loss, gh, gW, ws = kd.full_kl_fwd_bwd(hs, Ws, ht, Wt, mask, xs.T, 0, err_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    lay = kd.full_kl_workspace_layout(N, d, xt.d, V, 0)
    assert int(lay.chunk) == 4096
    ctrl = ws[lay.off_ctrl: lay.off_ctrl + 16].cpu().numpy()
    nv = int(ctrl[4:8].view(np.int32)[0])
    got = dict(loss=float(loss.item()), n_valid=nv,
               grad_h=gh.cpu().numpy().astype(np.float64),
               grad_W=gW.cpu().numpy().astype(np.float64),
               rows=kd.workspace_view(ws, lay, "rows", N, torch.int32)[:nv].cpu().numpy(),
               lse=kd.workspace_view(ws, lay, "lse", N, torch.float32)[:nv].cpu().numpy(),
               loss_rows=kd.workspace_view(ws, lay, "loss_rows", N,
                                           torch.float32)[:nv].cpu().numpy())
    del gh, gW, ws
    check_whole_batch(xs, got, full)
    check_grad_W_rows(xs, got, full)
    rows = sample_rows(xs)
    ref = oracle.full_kl_sampled_rows(xs.h_f32(), xs.W_f32(), xt.h_f32(), xt.W_f32(), xs.mask,
                                      xs.T, rows)
    assert max_rel_err(got["grad_h"][rows], ref["grad_h"]) <= TOL["bf16"][1]
    check_sum_rule(xs, got, rounding=4.01)
    check_projection_identity(xs, got)
