"""GPU parity of the full-vocabulary (K = V) distillation loss
(kd_full_kl_fwd_bwd) with the fp64 oracle (oracle/full_kl_oracle.py): element
by element at sizes spanning several tiles, chunks and ragged tails; zero at
teacher = student; agreement with the top-K path when the cache holds the
whole vocabulary; sampled rows at the 201,088-word vocabulary."""
import numpy as np
import pytest

import oracle
from top_kl_loss_token_b300 import synth
from kd_testutil import TOL, max_rel_err

pytestmark = pytest.mark.gpu


def _bf16(a):
    return synth.bf16_bits_to_f32(synth.bf16_bits(np.asarray(a, dtype=np.float32)))


def _dev(a):
    import torch
    return torch.from_numpy(synth.bf16_bits(a).view(np.int16)).view(torch.bfloat16).cuda()


def _inputs(seed, N, d_s, d_t, V, w_std=0.02, mask_frac=0.0):
    rng = np.random.default_rng(seed)
    h_s = _bf16(rng.standard_normal((N, d_s)))
    W_s = _bf16(w_std * rng.standard_normal((V, d_s)))
    h_t = _bf16(rng.standard_normal((N, d_t)))
    W_t = _bf16(w_std * 1.5 * rng.standard_normal((V, d_t)))
    mask = None
    if mask_frac > 0:
        mask = (rng.random(N) >= mask_frac).astype(np.uint8)
    return h_s, W_s, h_t, W_t, mask


def _run(kd, h_s, W_s, h_t, W_t, mask, T, chunk=0):
    import torch
    m = None if mask is None else torch.from_numpy(mask).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    N, d_s = h_s.shape
    V, d_t = W_t.shape[0], h_t.shape[1]
    loss, gh, gW, ws = kd.full_kl_fwd_bwd(_dev(h_s), _dev(W_s), _dev(h_t), _dev(W_t), m, T, chunk,
                                          err_flags=err)
    torch.cuda.synchronize()
    lay = kd.full_kl_workspace_layout(N, d_s, d_t, V, chunk)
    ctrl = ws[lay.off_ctrl: lay.off_ctrl + 16].cpu().numpy()
    nv = int(ctrl[4:8].view(np.int32)[0])
    return dict(loss=float(loss.item()), grad_h=gh.cpu().numpy().astype(np.float64),
                grad_W=gW.cpu().numpy().astype(np.float64), err=int(err.item()), n_valid=nv,
                ws=ws, lay=lay,
                rows=kd.workspace_view(ws, lay, "rows", N, torch.int32)[:nv].cpu().numpy(),
                lse=kd.workspace_view(ws, lay, "lse", N, torch.float32)[:nv].cpu().numpy(),
                loss_rows=kd.workspace_view(ws, lay, "loss_rows", N, torch.float32)[:nv].cpu().numpy())


@pytest.mark.parametrize("chunk", [0, 256, 1000])
def test_parity_masked_ragged_two_widths(kd, chunk):
    # N = 600 (5 row tiles), V = 3000 (23.4 blocks of 128), teacher and student
    # of different widths, T = 2, 20 % of the rows masked
    h_s, W_s, h_t, W_t, mask = _inputs(31, 600, 256, 192, 3000, w_std=0.05, mask_frac=0.2)
    T = 2.0
    got = _run(kd, h_s, W_s, h_t, W_t, mask, T, chunk)
    ref = oracle.full_kl_fwd_bwd(h_s, W_s, h_t, W_t, mask, T)
    tl, tg = TOL["bf16"]
    assert got["err"] == 0 and got["n_valid"] == ref["n_valid"]
    assert abs(got["loss"] - ref["loss"]) <= tl * abs(ref["loss"])
    assert max_rel_err(got["grad_h"], ref["grad_h"]) <= tg
    assert max_rel_err(got["grad_W"], ref["grad_W"]) <= tg
    vr = np.nonzero(ref["valid"])[0]
    np.testing.assert_array_equal(got["rows"], vr)
    np.testing.assert_allclose(got["lse"], ref["lse_s"][vr], rtol=tl, atol=tl)
    np.testing.assert_allclose(got["loss_rows"], ref["loss_rows"][vr], rtol=10 * tl,
                               atol=10 * tl * abs(ref["loss"]))


def test_zero_when_student_equals_teacher(kd):
    h_s, W_s, _, _, _ = _inputs(32, 300, 128, 128, 1000, w_std=0.1)
    got = _run(kd, h_s, W_s, h_s, W_s, None, 1.0)
    assert got["err"] == 0
    assert abs(got["loss"]) <= 1e-6
    ref = oracle.full_kl_fwd_bwd(h_s, W_s, *_inputs(33, 300, 128, 128, 1000, w_std=0.1)[2:4],
                                 None, 1.0)
    # gradients vanish up to rounding, far below a typical gradient's size
    assert np.abs(got["grad_W"]).max() <= 1e-4 * np.abs(ref["grad_W"]).max()
    assert np.abs(got["grad_h"]).max() <= 1e-4 * np.abs(ref["grad_h"]).max()


def test_matches_the_top_k_path_with_the_whole_vocabulary(kd):
    # the top-K path with K = V and the teacher's logits as the cache must give
    # the same loss and gradients as the teacher computed in the same pass
    import torch
    h_s, W_s, h_t, W_t, mask = _inputs(34, 400, 128, 96, 2000, w_std=0.05, mask_frac=0.1)
    T = 1.5
    full = _run(kd, h_s, W_s, h_t, W_t, mask, T)
    zt = (h_t.astype(np.float64) @ W_t.astype(np.float64).T).astype(np.float32)
    idx = np.tile(np.arange(2000, dtype=np.int32), (400, 1))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    loss, gh, gW, _ = kd.fwd_bwd(_dev(h_s), _dev(W_s), torch.from_numpy(idx).cuda(),
                                 torch.from_numpy(zt).cuda(), torch.from_numpy(mask).cuda(), T,
                                 err_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert abs(loss.item() - full["loss"]) <= 1e-3 * abs(full["loss"])
    assert max_rel_err(gh.cpu().numpy(), full["grad_h"]) <= 2e-2
    assert max_rel_err(gW.cpu().numpy(), full["grad_W"]) <= 2e-2


@pytest.mark.slow
def test_full_vocabulary_sampled_rows(kd):
    N, d, V = 4096, 2880, 201088
    h_s, W_s, h_t, W_t, mask = _inputs(35, N, d, d, V, mask_frac=0.05)
    got = _run(kd, h_s, W_s, h_t, W_t, mask, 1.0)
    assert got["err"] == 0
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, N - 1], rng.choice(N, 40, replace=False)]))
    ref = oracle.full_kl_sampled_rows(h_s, W_s, h_t, W_t, mask, 1.0, rows)
    assert got["n_valid"] == ref["n_valid"]
    tl, tg = TOL["bf16"]
    pos = {int(r): i for i, r in enumerate(got["rows"])}
    v = ref["valid"]
    gi = np.array([pos[int(r)] for r in rows[v]])
    np.testing.assert_allclose(got["lse"][gi], ref["lse_s"][v], rtol=tl, atol=tl)
    np.testing.assert_allclose(got["loss_rows"][gi], ref["loss_rows"][v], rtol=10 * tl,
                               atol=10 * tl * float(np.abs(ref["loss_rows"][v]).max()))
    assert max_rel_err(got["grad_h"][rows], ref["grad_h"]) <= tg
    assert got["loss"] == pytest.approx(float(np.mean(got["loss_rows"].astype(np.float64))),
                                        rel=1e-6)


@pytest.mark.parametrize("chunk", [0, 256])
def test_gradient_tile_and_its_products(kd, chunk):
    # The last chunk's stored dL/dz_s against the oracle, element by element:
    # the two stored exponentials (bf16, up to 2^-8 relative each) and the
    # tile's own rounding stay inside 1.1 * 2^-7 (q + p) / (T N_valid).  Then
    # grad_h rows of that chunk and (single chunk) grad_W against fp64
    # products of the call's own tile, within 3e-5 of sum |G| |W|.
    import torch
    h_s, W_s, h_t, W_t, mask = _inputs(41, 600, 256, 192, 3000, w_std=0.05, mask_frac=0.2)
    T = 2.0
    got = _run(kd, h_s, W_s, h_t, W_t, mask, T, chunk)
    lay = got["lay"]
    cpad, ldg, V = int(lay.chunk_pad), int(lay.ld_g), W_s.shape[0]
    c = min(chunk if chunk > 0 else int(lay.chunk), 600)
    j = (got["n_valid"] - 1) // c
    row0, count = j * c, got["n_valid"] - j * c
    g = kd.workspace_view(got["ws"], lay, "g", cpad * ldg, torch.int16).cpu()
    g = g.view(torch.bfloat16).double().numpy().reshape(cpad, ldg)
    rows = got["rows"][row0:row0 + count]
    ref = oracle.full_kl_grad_logits(h_s, W_s, h_t, W_t, mask, T)
    scale = 1.0 / (T * ref["n_valid"])
    G_ref = ref["G"][rows]
    bound = 1.1 * 2.0 ** -7 * (ref["q"][rows] + ref["p"][rows]) * scale + 1e-30
    err = np.abs(g[:count, :V] - G_ref)
    assert np.all(err <= bound), float((err / bound).max())
    assert np.all(g[:count, V:] == 0.0)
    G = g[:count, :V]
    Wd = W_s.astype(np.float64)
    assert np.all(np.abs(got["grad_h"][rows] - G @ Wd) <= 3e-5 * (np.abs(G) @ np.abs(Wd)) + 1e-30)
    if row0 == 0:
        H = h_s.astype(np.float64)[rows]
        assert np.all(np.abs(got["grad_W"] - G.T @ H) <= 3e-5 * (np.abs(G).T @ np.abs(H)) + 1e-30)
