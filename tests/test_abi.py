"""Host-side checks of the C ABI: the library loads, exports every function the
headers declare, plans workspaces, and rejects bad arguments before touching
a GPU (these run without one)."""
import ctypes
import os
import re

import numpy as np
import pytest

import top_kl_loss_token_b300 as kd
from top_kl_loss_token_b300 import build as kd_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(kd.LIB_PATH):
        kd_build.build()
    return kd.load_library()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(kd_[a-z0-9_]+)\s*\(",
                             text, flags=re.M):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(lib):
    decl = declared_functions()
    assert decl == set(kd.EXPORTS), decl ^ set(kd.EXPORTS)
    for name in decl:
        assert hasattr(lib, name), name


def test_workspace_plan_is_linear_in_chunk_not_in_n_times_v(lib):
    # Extra memory is O(chunk * V + N * K): quadrupling N at a fixed chunk adds
    # only O(N K) bytes, not O(N V).
    V, d, K, c = 201088, 2880, 100, 8192
    a = kd.workspace_bytes(32768, d, V, K, c)
    b = kd.workspace_bytes(131072, d, V, K, c)
    assert b - a < (131072 - 32768) * (8 * K + 64)
    dense = 131072 * V * 2
    assert b < dense / 10
    lay = kd.workspace_layout(32768, d, V, K, c)
    assert lay.chunk == c and lay.chunk_pad == c and lay.n_pb == (V + 127) // 128
    offs = [getattr(lay, f[0]) for f in kd.WorkspaceLayout._fields_ if f[0].startswith("off_")]
    assert all(o % 256 == 0 for o in offs) and len(set(offs)) == len(offs)
    assert lay.total > max(offs)
    # the chunk's exponential tile comes last, so the loss alone stops before it
    assert lay.off_g == max(offs)
    assert lay.total - lay.off_g == c * ((V + 255) // 256 * 256) * 2
    fwd = kd.workspace_bytes(32768, d, V, K, c, loss_only=True)
    assert fwd == lay.off_g and fwd < a / 10


def test_default_chunk_splits_evenly(lib):
    assert kd.default_chunk(32768, 2880, 201088) == 8192
    # the chunk's hidden states within 48 MiB of L2: at most 6144 tokens at
    # d = 4096, made equal (6 chunks of 32K tokens)
    assert kd.default_chunk(32768, 4096, 151936) == 5504
    assert kd.default_chunk(32768, 3072, 128256) == 8192
    c = kd.default_chunk(131072, 2880, 201088)
    assert c % 128 == 0 and c * 2 * ((201088 + 255) // 256 * 256) <= 4 << 30
    assert kd.default_chunk(64, 64, 512, kd.KD_FP32) == 128


def test_default_chunk_rule_over_many_sizes(lib):
    # the rule kd_topk_kl.h and kd_full_kl.h state: equal chunks of a multiple
    # of 128 rows, at most 8192, the vocabulary buffers within their budget,
    # and the chunk's hidden states within 48 MiB (unless one 128-row chunk is
    # already more)
    rng = np.random.default_rng(0)
    l2 = 48 << 20
    for _ in range(300):
        N = int(rng.integers(1, 300000))
        d = int(rng.integers(1, 1024)) * 8
        V = int(rng.integers(1, 400000))
        ldg = -(-V // 256) * 256
        for dt, elem in ((kd.KD_BF16, 2), (kd.KD_FP32, 4)):
            c = kd.default_chunk(N, d, V, dt)
            assert c % 128 == 0 and 128 <= c <= 8192, (N, d, V, c)
            pieces = -(-N // c)
            assert c - 128 < -(-N // pieces) <= c            # equal chunks
            assert c == 128 or c * d * elem <= l2, (N, d, V, c)
            assert c == 128 or c * ldg * elem <= 4 << 30
        dt_ = int(rng.integers(1, 1024)) * 8
        cf = lib.kd_full_kl_default_chunk(N, d, dt_, V)
        assert cf % 128 == 0 and 128 <= cf <= 8192
        assert cf == 128 or cf * (d + dt_) * 2 <= l2, (N, d, dt_, V, cf)
        assert cf == 128 or 2 * cf * ldg * 2 <= 8 << 30


def call_fwd_bwd(lib, **kw):
    args = dict(h=16, W=16, dtype=kd.KD_BF16, idx=16, logit=16, mask=None, N=8, d=16, V=32, K=4,
                T=1.0, chunk=0, loss=16, gh=16, gW=16, ws=16, ws_bytes=1 << 40, err=None, stream=None)
    args.update(kw)
    return lib.kd_topk_kl_fwd_bwd(args["h"], args["W"], args["dtype"], args["idx"], args["logit"],
                                  args["mask"], args["N"], args["d"], args["V"], args["K"],
                                  args["T"], args["chunk"], args["loss"], args["gh"], args["gW"],
                                  args["ws"], args["ws_bytes"], args["err"], args["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(W=None), 1), (dict(loss=None), 1), (dict(h=None), 1), (dict(gh=None), 1),
    (dict(N=-1), 1), (dict(d=0), 1), (dict(V=0), 1), (dict(K=0), 1),
    (dict(K=kd.KD_MAX_K + 1), 2), (dict(T=0.0), 1), (dict(T=float("nan")), 1),
    (dict(T=float("inf")), 1), (dict(T=-1.0), 1), (dict(d=12), 2), (dict(dtype=7), 1),
    (dict(dtype=kd.KD_FP32, d=6), 2), (dict(ws=None), 3), (dict(ws_bytes=100), 3),
    (dict(W=24), 1), (dict(ws=40), 3),
])
def test_host_side_argument_errors(lib, kw, status):
    assert call_fwd_bwd(lib, **kw) == status


def test_status_strings(lib):
    for s in range(5):
        assert lib.kd_status_string(s)
    assert kd.status_string(3) == "workspace missing or too small"


def test_umma_gemm_argument_errors(lib):
    f = lib.kd_umma_gemm_bf16
    assert f(16, 16, 16, 0, 8, 8, 0, 0, 0, 16, 16, None) == 1
    assert f(16, 16, 16, 8, 8, 12, 0, 0, 0, 16, 16, None) == 2   # K-major A with K % 8 != 0
    assert f(16, 16, 16, 12, 8, 8, 1, 0, 0, 16, 16, None) == 2   # MN-major A with M % 8 != 0
    assert f(None, 16, 16, 8, 8, 8, 0, 0, 0, 16, 16, None) == 1


def test_build_flags_target_sm103a():
    assert "arch=compute_103a,code=sm_103a" in kd_build.ARCH


def test_topk_cache_argument_errors_and_plan(lib):
    f = lib.kd_topk_cache_build
    ok = dict(h=256, W=256, N=8, d=16, V=300, K=4, chunk=0, idx=256, val=256, ws=256,
              ws_bytes=1 << 40)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(a["h"], a["W"], a["N"], a["d"], a["V"], a["K"], a["chunk"], a["idx"], a["val"],
                 a["ws"], a["ws_bytes"], None, None)
    assert call(W=None) == 1
    assert call(h=None) == 1
    assert call(K=0) == 1
    assert call(K=301) == 1              # K > V
    assert call(N=-1) == 1
    assert call(d=12) == 2               # rows must be 16-byte multiples
    assert call(K=kd.KD_MAX_K + 1, V=10 ** 6) == 2
    assert call(ws=None) == 3
    assert call(ws_bytes=10) == 3
    assert call(h=264) == 1              # misaligned
    # candidates are bounded by 128 K per row, block keys by V / 128 per row
    n = kd.topk_cache_workspace_bytes(8192, 2880, 201088, 100, 8192)
    per_row = 8 * (128 * 100 + 1571 + 1) + 8
    assert 8192 * per_row <= n <= 8192 * per_row + 4096
    assert lib.kd_topk_cache_default_chunk(32768, 201088, 100) % 128 == 0


def test_full_kl_argument_errors_and_plan(lib):
    f = lib.kd_full_kl_fwd_bwd
    ok = dict(hs=256, Ws=256, ht=256, Wt=256, mask=None, N=8, ds=16, dt=24, V=300, T=1.0,
              chunk=0, loss=256, gh=256, gW=256, ws=256, ws_bytes=1 << 40)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(a["hs"], a["Ws"], a["ht"], a["Wt"], a["mask"], a["N"], a["ds"], a["dt"], a["V"],
                 a["T"], a["chunk"], a["loss"], a["gh"], a["gW"], a["ws"], a["ws_bytes"], None, None)
    for kw in (dict(Ws=None), dict(Wt=None), dict(hs=None), dict(ht=None), dict(loss=None),
               dict(gh=None), dict(gW=None), dict(N=-1), dict(ds=0), dict(dt=0), dict(V=0),
               dict(T=0.0), dict(T=float("nan")), dict(T=-2.0), dict(ht=264)):
        assert call(**kw) == 1, kw
    assert call(ds=12) == 2 and call(dt=20) == 2
    assert call(ws=None) == 3 and call(ws_bytes=100) == 3
    # extra memory is O(chunk V + N): both models' exponential tiles per chunk
    a = kd.full_kl_workspace_bytes(32768, 2880, 2880, 201088, 8192)
    b = kd.full_kl_workspace_bytes(131072, 2880, 2880, 201088, 8192)
    assert b - a < (131072 - 32768) * 64
    assert a < 2 * 8192 * 201216 * 2 * 1.2
    lay = kd.full_kl_workspace_layout(32768, 2880, 2880, 201088, 8192)
    assert lay.chunk == 8192 and lay.off_idx_sorted == 0 and lay.off_rows > 0
    # both models' hidden states of a chunk within 48 MiB of L2: 4096 tokens
    # at d_s = d_t = 2880 (8 equal chunks of 32K tokens)
    assert lib.kd_full_kl_default_chunk(32768, 2880, 2880, 201088) == 4096
    assert lib.kd_full_kl_default_chunk(1000, 64, 64, 5000) == 1024


def test_bounded_wait_test_entry_rejects_bad_arguments(lib):
    f = lib.kd_umma_gemm_bf16_wait_test
    assert f(None, 16, 16, 8, 8, 8, 1000, 16, 16, None) == 1
    assert f(16, 16, 16, 8, 8, 8, 0, 16, 16, None) == 1      # a zero time limit
    assert f(16, 16, 16, 8, 8, 12, 1000, 16, 16, None) == 2  # K % 8 != 0


def test_product_path_fails_loudly_without_the_library(tmp_path):
    # A copy of the package without libkd_topk_kl.so: loading the library
    # raises, and the loss refuses host tensors before reaching it -- there is
    # no CPU or PyTorch fallback to land on.
    import shutil
    import subprocess
    import sys
    src = os.path.join(ROOT, "top_kl_loss_token_b300")
    shutil.copytree(src, tmp_path / "top_kl_loss_token_b300",
                    ignore=shutil.ignore_patterns("*.so", "*.so.tmp", "__pycache__", "_build"))
    code = (
        "import torch\n"
        "import top_kl_loss_token_b300 as kd\n"
        "for f in (lambda: kd.load_library(),\n"
        "          lambda: kd.fwd_bwd(torch.zeros(4, 8, dtype=torch.bfloat16),\n"
        "                             torch.zeros(16, 8, dtype=torch.bfloat16),\n"
        "                             torch.zeros(4, 2, dtype=torch.int32), torch.zeros(4, 2),\n"
        "                             None, 1.0)):\n"
        "    try:\n"
        "        f()\n"
        "        print('no error')\n"
        "    except Exception as e:\n"
        "        print(type(e).__name__, e)\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=tmp_path, capture_output=True, text=True,
                       timeout=300)
    lines = r.stdout.strip().splitlines()
    assert len(lines) == 2, r.stdout + r.stderr
    assert lines[0].startswith("RuntimeError") and "is missing" in lines[0], lines[0]
    assert lines[1].startswith("ValueError") and "CUDA tensor" in lines[1], lines[1]


def test_workspace_size_checks_of_the_two_calls(lib):
    # Host-side rejections only (they return before any CUDA call): the loss
    # alone needs kd_topk_kl_fwd_workspace_bytes, fwd+bwd the full size.
    N, d, V, K = 64, 16, 1000, 4
    full = kd.workspace_bytes(N, d, V, K)
    fwd = kd.workspace_bytes(N, d, V, K, loss_only=True)
    assert 0 < fwd < full
    assert call_fwd_bwd(lib, N=N, d=d, V=V, K=K, ws=256, ws_bytes=fwd) == 3
    assert call_fwd_bwd(lib, N=N, d=d, V=V, K=K, ws=256, ws_bytes=full - 1) == 3
    st = lib.kd_topk_kl_fwd(16, 16, kd.KD_BF16, 16, 16, None, N, d, V, K, 1.0, 0, 16, 256,
                            fwd - 1, None, None)
    assert st == 3
