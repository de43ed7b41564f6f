"""Helpers shared by the GPU tests: moving a synthetic problem to the device,
running the library, and the parity tolerances.

Tolerances (fixed by the target): bf16 inputs -> loss relative error <= 1e-3
and gradient max-abs error <= 2e-2 * max|gradient|; fp32 inputs -> 1e-5 and
1e-4."""
import importlib.util
import os

import numpy as np

TOL = {"bf16": (1e-3, 2e-2), "fp32": (1e-5, 1e-4)}

_HERE = os.path.dirname(os.path.abspath(__file__))


def fullsize_oracle(cfg, x):
    """The fp64 oracle's whole-batch forward (loss, every lse and loss term)
    and sampled grad_W rows for full-size config cfg, from the local cache
    that tests/golden/make_fullsize_oracle.py writes (computed now, and
    cached, when it is missing or was made from other inputs)."""
    spec = importlib.util.spec_from_file_location(
        "make_fullsize_oracle", os.path.join(_HERE, "golden", "make_fullsize_oracle.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.load_or_compute(cfg, x)


def fullsize_full_oracle(cfg, xs, xt):
    """The full-vocabulary oracle's whole-batch forward and sampled grad_W rows
    for student xs and teacher xt (config cfg's sizes), from the same local
    cache (computed now, and cached, when missing or made from other inputs)."""
    spec = importlib.util.spec_from_file_location(
        "make_fullsize_oracle", os.path.join(_HERE, "golden", "make_fullsize_oracle.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.load_or_compute_full(cfg, xs, xt)


def to_device(x, device="cuda"):
    import torch
    if x.dtype == "bf16":
        h = torch.from_numpy(x.h.view(np.int16)).view(torch.bfloat16).to(device)
        W = torch.from_numpy(x.W.view(np.int16)).view(torch.bfloat16).to(device)
    else:
        h = torch.from_numpy(x.h).to(device)
        W = torch.from_numpy(x.W).to(device)
    idx = torch.from_numpy(x.idx).to(device)
    logit = torch.from_numpy(x.logit).to(device)
    mask = None if x.mask is None else torch.from_numpy(x.mask).to(device)
    return h, W, idx, logit, mask


def run_gpu(kd, x, chunk=0, want_grads=True, tensors=None):
    import torch
    h, W, idx, logit, mask = tensors if tensors is not None else to_device(x)
    err = torch.zeros(1, dtype=torch.int32, device=h.device)
    if want_grads:
        loss, gh, gW, ws = kd.fwd_bwd(h, W, idx, logit, mask, x.T, chunk, err_flags=err)
    else:
        loss, ws = kd.fwd(h, W, idx, logit, mask, x.T, chunk, err_flags=err)
        gh = gW = None
    torch.cuda.synchronize()
    N, d, V, K = x.N, x.d, x.V, x.K
    lay = kd.workspace_layout(N, d, V, K, chunk, kd.KD_BF16 if x.dtype == "bf16" else kd.KD_FP32)
    ctrl = ws[lay.off_ctrl: lay.off_ctrl + 16].cpu().numpy()
    n_valid = int(ctrl[4:8].view(np.int32)[0])
    out = dict(
        loss=float(loss.item()),
        grad_h=None if gh is None else gh.cpu().numpy().astype(np.float64),
        grad_W=None if gW is None else gW.cpu().numpy().astype(np.float64),
        err=int(err.item()),
        n_valid=n_valid,
        rows=kd.workspace_view(ws, lay, "rows", N, torch.int32)[:n_valid].cpu().numpy(),
        lse=kd.workspace_view(ws, lay, "lse", N, torch.float32)[:n_valid].cpu().numpy(),
        loss_rows=kd.workspace_view(ws, lay, "loss_rows", N, torch.float32)[:n_valid].cpu().numpy(),
        ws=ws,
        lay=lay,
    )
    return out


def max_rel_err(got, want):
    scale = float(np.abs(want).max())
    if scale == 0.0:
        return float(np.abs(got).max())
    return float(np.abs(got - want).max()) / scale


def assert_parity(got, ref, dtype, grads=True):
    tl, tg = TOL[dtype]
    lerr = abs(got["loss"] - ref["loss"]) / max(abs(ref["loss"]), 1e-30)
    assert lerr <= tl, f"loss {got['loss']} vs {ref['loss']} (rel {lerr:.3e})"
    if grads:
        eh = max_rel_err(got["grad_h"], ref["grad_h"])
        ew = max_rel_err(got["grad_W"], ref["grad_W"])
        assert eh <= tg, f"grad_h max-abs error {eh:.3e} of max|grad_h|"
        assert ew <= tg, f"grad_W max-abs error {ew:.3e} of max|grad_W|"
        return lerr, eh, ew
    return lerr, None, None
