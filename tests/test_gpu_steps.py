"""Step-by-step GPU parity: the intermediates that one kd_topk_kl_fwd_bwd call
leaves in its workspace (layout and contents in kd_topk_kl_steps.h), each
compared with the fp64 oracle on its own:

  teacher preparation   sorted entries, probabilities, sum p ln p, sum p;
  block offsets         where each 128-column vocabulary block starts in a
                        row's sorted entries (exact);
  gradient tile         dL/dz of the last chunk, element by element, within
                        the rounding of its storage type (bf16: 8-bit
                        significand);
  gradient products     grad_h = G W and grad_W = G^T h against fp64 products
                        of the call's own G, which separates the contractions
                        from the rounding of G.
"""
import numpy as np
import pytest

import oracle
from top_kl_loss_token_b300 import synth
from kd_testutil import run_gpu

pytestmark = pytest.mark.gpu

NO_INDEX = 0x7FFFFFFF


def region(kd, got, name, count, dtype):
    return kd.workspace_view(got["ws"], got["lay"], name, count, dtype).cpu().numpy()


def last_chunk(got, chunk, N):
    """(first compacted row, count) of the last chunk that holds valid rows."""
    c = chunk if chunk > 0 else int(got["lay"].chunk)
    c = min(c, N)
    j = (got["n_valid"] - 1) // c
    return j * c, got["n_valid"] - j * c


def row_alpha(kd, got, N, row0, count):
    """alpha_i of the chunk rows row0 .. row0 + count (bf16 with gradients)."""
    import torch
    rs = region(kd, got, "rowstat", 4 * N, torch.float32)
    return rs[2 * N + row0: 2 * N + row0 + count].astype(np.float64)


def stored_tile(kd, got, dtype, N, row0, count, cpad, ldg):
    """The last chunk's dL/dz [count, ldg] as the workspace holds it: fp32
    itself, or (bf16) the stored values times the row factor alpha_i."""
    import torch
    if dtype == "bf16":
        g = region(kd, got, "g", cpad * ldg, torch.int16)
        g = torch.from_numpy(g).view(torch.bfloat16).double().numpy().reshape(cpad, ldg)[:count]
        return g * row_alpha(kd, got, N, row0, count)[:, None]
    g = region(kd, got, "g", cpad * ldg, torch.float32).astype(np.float64).reshape(cpad, ldg)
    return g[:count]


def teacher_case(K=16):
    # duplicates, out-of-range indices and -inf logits in valid rows, plus masked rows
    x = synth.make_inputs(300, 64, 1100, K, T=1.5, dtype="bf16", seed=201, mask="random0.2")
    rng = np.random.default_rng(7)
    x.mask[:12] = 1
    x.idx[0, 3] = x.idx[0, 5]
    x.idx[1, :4] = x.idx[1, 4]
    x.idx[2, 7] = 1100
    x.idx[3, 0] = -1
    x.logit[4, 2] = -np.inf
    x.idx[5] = rng.integers(0, 20, size=K)
    return x


# K <= 128 runs one warp per row (entries in registers, 1, 2 or 4 per lane);
# larger K one block per row with the entries in shared memory
@pytest.mark.parametrize("K", [16, 9, 33, 100, 128, 200])
def test_teacher_preparation(kd, K):
    import torch
    x = teacher_case(K)
    got = run_gpu(kd, x, want_grads=False)
    assert got["err"] == oracle.FLAG_INDEX_RANGE
    N, K, V = x.N, x.K, x.V
    p_ref, valid, _ = oracle.teacher_distribution(x.idx, x.logit, x.mask, V, x.T)
    idx_s = region(kd, got, "idx_sorted", N * K, torch.int32).reshape(N, K)
    p_s = region(kd, got, "p_sorted", N * K, torch.float32).reshape(N, K)
    plogp = region(kd, got, "plogp", N, torch.float32)
    psum = region(kd, got, "psum", N, torch.float32)
    plogp_ref = oracle.teacher_plogp(p_ref)
    for r in np.nonzero(valid)[0]:
        keep = (x.idx[r] >= 0) & (x.idx[r] < V)
        n = int(keep.sum())
        # the same multiset of (index, p) pairs; order by index, then by p
        want = sorted(zip(x.idx[r][keep].tolist(), p_ref[r][keep].tolist()))
        have = sorted(zip(idx_s[r, :n].tolist(), p_s[r, :n].tolist()))
        assert [a for a, _ in have] == [a for a, _ in want], r
        np.testing.assert_array_equal(idx_s[r, :n], np.sort(x.idx[r][keep]))
        np.testing.assert_allclose([b for _, b in have], [b for _, b in want],
                                   rtol=2e-6, atol=1e-12, err_msg=str(r))
        assert np.all(idx_s[r, n:] == NO_INDEX) and np.all(p_s[r, n:] == 0.0)
        assert plogp[r] == pytest.approx(plogp_ref[r], rel=1e-5, abs=1e-6)
        assert psum[r] == pytest.approx(1.0, abs=2e-6)


@pytest.mark.parametrize("chunk", [0, 128])
def test_block_offsets(kd, chunk):
    import torch
    x = teacher_case()
    got = run_gpu(kd, x, chunk, want_grads=False)
    lay = got["lay"]
    N, K = x.N, x.K
    n_pb, cpad = int(lay.n_pb), int(lay.chunk_pad)
    row0, count = last_chunk(got, chunk, N)
    boff = region(kd, got, "boff", (n_pb + 1) * cpad, torch.int16).view(np.uint16)
    boff = boff.reshape(n_pb + 1, cpad).astype(np.int64)
    idx_s = region(kd, got, "idx_sorted", N * K, torch.int32).reshape(N, K).astype(np.int64)
    starts = np.arange(n_pb + 1) * 128
    for i in range(count):
        r = got["rows"][row0 + i]
        keep = (x.idx[r] >= 0) & (x.idx[r] < x.V)
        ref = np.searchsorted(np.sort(x.idx[r][keep]), starts, side="left")
        np.testing.assert_array_equal(boff[:, i], ref, err_msg=str(i))
        np.testing.assert_array_equal(boff[:, i], np.searchsorted(idx_s[r], starts, side="left"))


def grad_tile_bound(G_ref, x, valid_rows, n_valid):
    """What the per-element error bound of the stored G is built from: the
    softmax part q / (T N) passes through the rounding of the stored
    exponential (bf16: up to 2^-8 relative, 8-bit significand) and G itself
    through one more rounding (2^-8 |G| <= 2^-8 (q + p) / (T N)), so the
    total stays inside 1.1 * 2^-7 (q + p) / (T N).  Returns q, the scattered
    teacher probabilities p and 1 / (T N_valid)."""
    scale = 1.0 / (x.T * n_valid)
    P = np.zeros_like(G_ref)
    idx = x.idx[valid_rows].astype(np.int64)
    keep = (idx >= 0) & (idx < x.V)
    p, _, _ = oracle.teacher_distribution(x.idx, x.logit, x.mask, x.V, x.T)
    rr = np.repeat(np.arange(len(valid_rows)), x.K).reshape(idx.shape)
    np.add.at(P, (rr[keep], idx[keep]), p[valid_rows][keep])
    q = G_ref / scale + P
    return q, P, scale


@pytest.mark.parametrize("dtype,chunk", [("bf16", 0), ("bf16", 256), ("fp32", 0)])
def test_gradient_tile(kd, dtype, chunk):
    import torch
    if dtype == "bf16":
        x = synth.make_inputs(600, 256, 3000, 16, T=2.0, dtype="bf16", seed=202,
                              mask="random0.2")
    else:
        x = synth.make_inputs(150, 20, 300, 7, T=2.0, dtype="fp32", seed=203,
                              mask="random0.25", w_std=0.3)
    got = run_gpu(kd, x, chunk)
    lay = got["lay"]
    cpad, ldg = int(lay.chunk_pad), int(lay.ld_g)
    row0, count = last_chunk(got, chunk, x.N)
    g = stored_tile(kd, got, dtype, x.N, row0, count, cpad, ldg)
    rows = got["rows"][row0:row0 + count]
    ref = oracle.grad_logits(x.h_f32(), x.W_f32(), x.idx, x.logit, x.mask, x.T)
    G_ref = ref["G"][rows]
    q, P, scale = grad_tile_bound(G_ref, x, rows, ref["n_valid"])
    rel = 1.1 * 2.0 ** -7 if dtype == "bf16" else 2e-5
    err = np.abs(g[:count, :x.V] - G_ref)
    bound = rel * (q + P) * scale + 1e-30
    worst = np.unravel_index(np.argmax(err / bound), err.shape)
    assert np.all(err <= bound), (worst, g[:count, :x.V][worst], G_ref[worst], bound[worst])
    assert np.all(g[:count, x.V:] == 0.0)
    # every valid row of dL/dz sums to zero (softmax and p both sum to one),
    # up to the summed bound above: rel * 2 / (T N)
    assert np.abs(g[:count, :x.V].sum(axis=1)).max() <= 2.2 * rel * scale


@pytest.mark.parametrize("dtype,chunk", [("bf16", 0), ("bf16", 256), ("fp32", 0)])
def test_gradient_products_of_the_stored_tile(kd, dtype, chunk):
    """grad_h rows of the last chunk = G W, and (single chunk) grad_W = G^T h,
    against fp64 products of the call's own G: only the fp32 accumulation of
    the contractions remains, bounded by 3e-5 of sum |G| |W| per element."""
    import torch
    if dtype == "bf16":
        x = synth.make_inputs(600, 256, 3000, 16, T=2.0, dtype="bf16", seed=204,
                              mask="random0.2")
    else:
        x = synth.make_inputs(150, 20, 300, 7, T=2.0, dtype="fp32", seed=205,
                              mask="random0.25", w_std=0.3)
    got = run_gpu(kd, x, chunk)
    lay = got["lay"]
    cpad, ldg = int(lay.chunk_pad), int(lay.ld_g)
    row0, count = last_chunk(got, chunk, x.N)
    rows = got["rows"][row0:row0 + count]
    W = x.W_f32().astype(np.float64)
    if dtype == "bf16":
        # the stored operands of the products: g' (dL/dz = alpha g') and the
        # chunk's h rows scaled by alpha (bf16): grad_h = alpha (g' W) and
        # grad_W = g'^T (alpha h)
        g = region(kd, got, "g", cpad * ldg, torch.int16)
        G = torch.from_numpy(g).view(torch.bfloat16).double().numpy().reshape(cpad, ldg)
        G = G[:count, :x.V]
        alpha = row_alpha(kd, got, x.N, row0, count)[:, None]
        hc = region(kd, got, "hc", cpad * x.d, torch.int16)
        H = torch.from_numpy(hc).view(torch.bfloat16).double().numpy().reshape(cpad, x.d)
        H = H[:count]
    else:
        g = region(kd, got, "g", cpad * ldg, torch.float32).astype(np.float64)
        G = g.reshape(cpad, ldg)[:count, :x.V]
        alpha = np.ones((count, 1))
        H = x.h_f32().astype(np.float64)[rows]
    want_h = alpha * (G @ W)
    bound_h = 3e-5 * (np.abs(alpha * G) @ np.abs(W)) + 1e-30
    assert np.all(np.abs(got["grad_h"][rows] - want_h) <= bound_h)
    masked = np.setdiff1d(np.arange(x.N), got["rows"])
    assert np.all(got["grad_h"][masked] == 0.0)
    if row0 == 0:  # a single chunk: grad_W is this tile's product alone
        want_W = G.T @ H
        bound_W = 3e-5 * (np.abs(G).T @ np.abs(H)) + 1e-30
        assert np.all(np.abs(got["grad_W"] - want_W) <= bound_W)
        if dtype == "bf16":
            # and the scaled rows are alpha h rounded once to bf16
            h_ref = alpha * x.h_f32().astype(np.float64)[rows]
            assert np.all(np.abs(H - h_ref) <= 2.0 ** -8 * np.abs(h_ref))
