"""Fused chunked top-K KL distillation loss for B300 (sm_103a).

Python binding of the C ABI in include/kd_topk_kl.h and
include/kd_topk_kl_steps.h.  It only marshals arguments: torch provides the
device memory and the stream, every step runs in the CUDA kernels of
libkd_topk_kl.so.  There is no other implementation behind these functions;
if the library is missing they raise.

The loss is the KL divergence of a student against an offline teacher cache
of the top K (index, logit) pairs per position ("Efficient Knowledge
Distillation for LLMs: Offline Top-K Logits and a Fused Chunked KL Loss",
ai2day.live story, "What did the researchers change?"), computed chunk by
chunk over the tokens without materialising the N x V logit grid.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libkd_topk_kl.so")

KD_BF16 = 0
KD_FP32 = 1
KD_FLAG_INDEX_RANGE = 1
KD_FLAG_BAD_TEACHER = 2
KD_FLAG_TIMEOUT = 4
KD_FLAG_INTERNAL = 8
KD_MAX_K = 4096

STATUS = {0: "KD_OK", 1: "KD_ERR_INVALID_ARG", 2: "KD_ERR_UNSUPPORTED", 3: "KD_ERR_WORKSPACE",
          4: "KD_ERR_CUDA"}

# Every symbol the headers declare.
EXPORTS = ["kd_topk_kl_workspace_bytes", "kd_topk_kl_fwd_workspace_bytes",
           "kd_topk_kl_default_chunk", "kd_topk_kl_fwd_bwd",
           "kd_topk_kl_fwd", "kd_status_string", "kd_topk_kl_workspace_layout",
           "kd_umma_gemm_bf16", "kd_timing_enable", "kd_timing_collect",
           "kd_topk_kl_fwd_bwd_noalloc", "kd_topk_cache_workspace_bytes",
           "kd_topk_cache_default_chunk", "kd_topk_cache_build", "kd_umma_gemm_bf16_wait_test",
           "kd_full_kl_workspace_bytes", "kd_full_kl_default_chunk", "kd_full_kl_fwd_bwd",
           "kd_full_kl_workspace_layout", "kd_topk_kl_prepare", "kd_topk_kl_fwd_bwd_prepared",
           "kd_topk_kl_fwd_prepared"]

# Size of the library-held scratch array used by kd_topk_kl_fwd_bwd_noalloc.
KD_NOALLOC_SCRATCH_BYTES = 64 << 20

_LIB = None


class KDError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}")
        self.status = status


class WorkspaceLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("chunk", "chunk_pad", "n_pb", "ld_g")] + [
        (n, ctypes.c_size_t) for n in (
            "off_ctrl", "off_row_ok", "off_rows", "off_idx_sorted", "off_p_sorted", "off_plogp",
            "off_psum", "off_lse", "off_loss_rows", "off_part_m", "off_part_l", "off_part_ps",
            "off_boff", "off_top1", "off_rowstat", "off_hc", "off_g", "off_sched", "total")]


class TimingEntry(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int64),
                ("total_ms", ctypes.c_double)]


def load_library(path: str = LIB_PATH):
    """Loads libkd_topk_kl.so (raises if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m top_kl_loss_token_b300.build`")
    lib = ctypes.CDLL(path)
    i64, i32, f32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p
    sz = ctypes.c_size_t
    lib.kd_topk_kl_workspace_bytes.argtypes = [i64, i64, i64, i32, i64, ctypes.c_int]
    lib.kd_topk_kl_workspace_bytes.restype = sz
    lib.kd_topk_kl_fwd_workspace_bytes.argtypes = [i64, i64, i64, i32, i64, ctypes.c_int]
    lib.kd_topk_kl_fwd_workspace_bytes.restype = sz
    lib.kd_topk_kl_default_chunk.argtypes = [i64, i64, i64, ctypes.c_int]
    lib.kd_topk_kl_default_chunk.restype = i64
    lib.kd_topk_kl_workspace_layout.argtypes = [i64, i64, i64, i32, i64, ctypes.c_int,
                                                ctypes.POINTER(WorkspaceLayout)]
    lib.kd_topk_kl_workspace_layout.restype = ctypes.c_int
    lib.kd_topk_kl_fwd_bwd.argtypes = [vp, vp, ctypes.c_int, vp, vp, vp, i64, i64, i64, i32, f32,
                                       i64, vp, vp, vp, vp, sz, vp, vp]
    lib.kd_topk_kl_fwd_bwd.restype = ctypes.c_int
    lib.kd_topk_kl_fwd.argtypes = [vp, vp, ctypes.c_int, vp, vp, vp, i64, i64, i64, i32, f32, i64,
                                   vp, vp, sz, vp, vp]
    lib.kd_topk_kl_fwd.restype = ctypes.c_int
    lib.kd_topk_kl_prepare.argtypes = [vp, vp, vp, i64, i64, i64, i32, f32, i64, ctypes.c_int,
                                       vp, sz, vp, vp, vp]
    lib.kd_topk_kl_prepare.restype = ctypes.c_int
    lib.kd_topk_kl_fwd_bwd_prepared.argtypes = [vp, vp, ctypes.c_int, i64, i64, i64, i32, f32,
                                                i64, vp, vp, vp, vp, vp, sz, vp, vp]
    lib.kd_topk_kl_fwd_bwd_prepared.restype = ctypes.c_int
    lib.kd_topk_kl_fwd_prepared.argtypes = [vp, vp, ctypes.c_int, i64, i64, i64, i32, f32, i64,
                                            vp, vp, vp, sz, vp, vp]
    lib.kd_topk_kl_fwd_prepared.restype = ctypes.c_int
    lib.kd_topk_kl_fwd_bwd_noalloc.argtypes = [vp, vp, ctypes.c_int, vp, vp, vp, i64, i64, i64,
                                               i32, f32, i64, vp, vp, vp, vp, vp]
    lib.kd_topk_kl_fwd_bwd_noalloc.restype = ctypes.c_int
    lib.kd_topk_cache_workspace_bytes.argtypes = [i64, i64, i64, i32, i64]
    lib.kd_topk_cache_workspace_bytes.restype = sz
    lib.kd_topk_cache_default_chunk.argtypes = [i64, i64, i32]
    lib.kd_topk_cache_default_chunk.restype = i64
    lib.kd_topk_cache_build.argtypes = [vp, vp, i64, i64, i64, i32, i64, vp, vp, vp, sz, vp, vp]
    lib.kd_topk_cache_build.restype = ctypes.c_int
    lib.kd_full_kl_workspace_bytes.argtypes = [i64, i64, i64, i64, i64]
    lib.kd_full_kl_workspace_bytes.restype = sz
    lib.kd_full_kl_default_chunk.argtypes = [i64, i64, i64, i64]
    lib.kd_full_kl_default_chunk.restype = i64
    lib.kd_full_kl_workspace_layout.argtypes = [i64, i64, i64, i64, i64,
                                                ctypes.POINTER(WorkspaceLayout)]
    lib.kd_full_kl_workspace_layout.restype = ctypes.c_int
    lib.kd_full_kl_fwd_bwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, f32, i64, vp, vp,
                                       vp, vp, sz, vp, vp]
    lib.kd_full_kl_fwd_bwd.restype = ctypes.c_int
    lib.kd_status_string.argtypes = [ctypes.c_int]
    lib.kd_status_string.restype = ctypes.c_char_p
    lib.kd_umma_gemm_bf16.argtypes = [vp, vp, vp, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, vp, vp, vp]
    lib.kd_umma_gemm_bf16.restype = ctypes.c_int
    lib.kd_umma_gemm_bf16_wait_test.argtypes = [vp, vp, vp, i64, i64, i64, ctypes.c_uint32, vp, vp,
                                                vp]
    lib.kd_umma_gemm_bf16_wait_test.restype = ctypes.c_int
    lib.kd_timing_enable.argtypes = [ctypes.c_int]
    lib.kd_timing_enable.restype = ctypes.c_int
    lib.kd_timing_collect.argtypes = [ctypes.POINTER(TimingEntry), i32, ctypes.POINTER(i32)]
    lib.kd_timing_collect.restype = ctypes.c_int
    _LIB = lib
    return lib


def _check(st: int, where: str):
    if st != 0:
        raise KDError(st, where)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return KD_BF16
    if t.dtype == torch.float32:
        return KD_FP32
    raise TypeError(f"h and W must be bfloat16 or float32, got {t.dtype}")


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def workspace_bytes(N: int, d: int, V: int, K: int, chunk: int = 0, dtype: int = KD_BF16,
                    loss_only: bool = False) -> int:
    """Workspace bytes of kd_topk_kl_fwd_bwd, or with loss_only of kd_topk_kl_fwd."""
    lib = load_library()
    f = lib.kd_topk_kl_fwd_workspace_bytes if loss_only else lib.kd_topk_kl_workspace_bytes
    n = f(N, d, V, K, chunk, dtype)
    if n == 0:
        raise KDError(1, "kd_topk_kl_workspace_bytes")
    return int(n)


def default_chunk(N: int, d: int, V: int, dtype: int = KD_BF16) -> int:
    return int(load_library().kd_topk_kl_default_chunk(N, d, V, dtype))


def workspace_layout(N: int, d: int, V: int, K: int, chunk: int = 0,
                     dtype: int = KD_BF16) -> WorkspaceLayout:
    lay = WorkspaceLayout()
    _check(load_library().kd_topk_kl_workspace_layout(N, d, V, K, chunk, dtype, ctypes.byref(lay)),
           "kd_topk_kl_workspace_layout")
    return lay


def _validate(h, W, idx, logit, mask):
    import torch
    for name, t in (("h", h), ("W", W), ("topk_idx", idx), ("topk_logit", logit)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if h.dtype != W.dtype:
        raise TypeError("h and W must have the same dtype")
    if idx.dtype != torch.int32 or logit.dtype != torch.float32:
        raise TypeError("topk_idx must be int32 and topk_logit float32")
    if mask is not None and (mask.dtype != torch.uint8 or not mask.is_cuda
                             or not mask.is_contiguous()):
        raise TypeError("mask must be a contiguous uint8 CUDA tensor")
    N, d = h.shape
    V, d2 = W.shape
    if d2 != d or idx.shape != logit.shape or idx.shape[0] != N:
        raise ValueError("shape mismatch")
    if mask is not None and mask.shape != (N,):
        raise ValueError("mask must have shape [N]")
    return N, d, V, idx.shape[1]


def allocate_workspace(N, d, V, K, chunk=0, dtype=KD_BF16, device=None, loss_only=False):
    import torch
    n = workspace_bytes(N, d, V, K, chunk, dtype, loss_only)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def kd_topk_kl_fwd_bwd(h, W, topk_idx, topk_logit, mask=None, T: float = 1.0, chunk: int = 0,
                       loss=None, grad_h=None, grad_W=None, workspace=None, err_flags=None,
                       stream=None):
    """Loss, grad_h and grad_W of the top-K KL loss (see include/kd_topk_kl.h).

    Returns (loss [1] fp32, grad_h [N, d] fp32, grad_W [V, d] fp32, workspace).
    Asynchronous on the current (or given) stream."""
    import torch
    N, d, V, K = _validate(h, W, topk_idx, topk_logit, mask)
    dt = _dtype_code(h)
    dev = h.device
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=dev)
    if grad_h is None:
        grad_h = torch.empty((N, d), dtype=torch.float32, device=dev)
    if grad_W is None:
        grad_W = torch.empty((V, d), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = allocate_workspace(N, d, V, K, chunk, dt, dev)
    st = load_library().kd_topk_kl_fwd_bwd(
        _ptr(h), _ptr(W), dt, _ptr(topk_idx), _ptr(topk_logit), _ptr(mask), N, d, V, K,
        float(T), int(chunk), _ptr(loss), _ptr(grad_h), _ptr(grad_W), _ptr(workspace),
        workspace.numel(), _ptr(err_flags), _stream_handle(stream))
    _check(st, "kd_topk_kl_fwd_bwd")
    return loss, grad_h, grad_W, workspace


def kd_topk_kl_fwd(h, W, topk_idx, topk_logit, mask=None, T: float = 1.0, chunk: int = 0,
                   loss=None, workspace=None, err_flags=None, stream=None):
    """The loss alone.  Returns (loss [1] fp32, workspace)."""
    import torch
    N, d, V, K = _validate(h, W, topk_idx, topk_logit, mask)
    dt = _dtype_code(h)
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=h.device)
    if workspace is None:
        workspace = allocate_workspace(N, d, V, K, chunk, dt, h.device, loss_only=True)
    st = load_library().kd_topk_kl_fwd(
        _ptr(h), _ptr(W), dt, _ptr(topk_idx), _ptr(topk_logit), _ptr(mask), N, d, V, K,
        float(T), int(chunk), _ptr(loss), _ptr(workspace), workspace.numel(), _ptr(err_flags),
        _stream_handle(stream))
    _check(st, "kd_topk_kl_fwd")
    return loss, workspace


def kd_topk_kl_fwd_bwd_noalloc(h, W, topk_idx, topk_logit, loss, grad_h, grad_W, mask=None,
                               T: float = 1.0, chunk: int = 0, err_flags=None, stream=None):
    """kd_topk_kl_fwd_bwd for callers that cannot allocate device memory (see
    include/kd_topk_kl.h): the workspace is the library's own fixed scratch
    array, and the caller passes the output tensors, so this function
    allocates nothing on the device.  Returns (loss, grad_h, grad_W)."""
    N, d, V, K = _validate(h, W, topk_idx, topk_logit, mask)
    dt = _dtype_code(h)
    for name, t, shape in (("loss", loss, (1,)), ("grad_h", grad_h, (N, d)),
                           ("grad_W", grad_W, (V, d))):
        if (not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != shape
                or t.element_size() != 4 or not t.is_floating_point()):
            raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor of shape {shape}")
        if t.device != h.device:
            raise ValueError(f"{name} is on {t.device}, the inputs on {h.device}")
    st = load_library().kd_topk_kl_fwd_bwd_noalloc(
        _ptr(h), _ptr(W), dt, _ptr(topk_idx), _ptr(topk_logit), _ptr(mask), N, d, V, K,
        float(T), int(chunk), _ptr(loss), _ptr(grad_h), _ptr(grad_W), _ptr(err_flags),
        _stream_handle(stream))
    _check(st, "kd_topk_kl_fwd_bwd_noalloc")
    return loss, grad_h, grad_W


def topk_cache_workspace_bytes(N: int, d: int, V: int, K: int, chunk: int = 0) -> int:
    n = load_library().kd_topk_cache_workspace_bytes(N, d, V, K, chunk)
    if n == 0:
        raise KDError(1, "kd_topk_cache_workspace_bytes")
    return int(n)


def kd_topk_cache_build(h, W, K: int, chunk: int = 0, topk_idx=None, topk_logit=None,
                        workspace=None, err_flags=None, stream=None):
    """The offline teacher top-K cache of teacher hidden states h [N, d] (bf16)
    against the teacher LM head W [V, d] (bf16); see include/kd_topk_cache.h.
    Returns (topk_idx [N, K] int32, topk_logit [N, K] fp32, workspace)."""
    import torch
    for name, t in (("h", h), ("W", W)):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be a contiguous bfloat16 CUDA tensor")
    N, d = h.shape
    V, d2 = W.shape
    if d2 != d:
        raise ValueError("shape mismatch")
    dev = h.device
    if topk_idx is None:
        topk_idx = torch.empty((N, K), dtype=torch.int32, device=dev)
    if topk_logit is None:
        topk_logit = torch.empty((N, K), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(topk_cache_workspace_bytes(N, d, V, K, chunk), dtype=torch.uint8,
                                device=dev)
    st = load_library().kd_topk_cache_build(
        _ptr(h), _ptr(W), N, d, V, int(K), int(chunk), _ptr(topk_idx), _ptr(topk_logit),
        _ptr(workspace), workspace.numel(), _ptr(err_flags), _stream_handle(stream))
    _check(st, "kd_topk_cache_build")
    return topk_idx, topk_logit, workspace


def full_kl_workspace_bytes(N: int, d_s: int, d_t: int, V: int, chunk: int = 0) -> int:
    n = load_library().kd_full_kl_workspace_bytes(N, d_s, d_t, V, chunk)
    if n == 0:
        raise KDError(1, "kd_full_kl_workspace_bytes")
    return int(n)


def full_kl_workspace_layout(N: int, d_s: int, d_t: int, V: int, chunk: int = 0) -> WorkspaceLayout:
    lay = WorkspaceLayout()
    _check(load_library().kd_full_kl_workspace_layout(N, d_s, d_t, V, chunk, ctypes.byref(lay)),
           "kd_full_kl_workspace_layout")
    return lay


def kd_full_kl_fwd_bwd(h_s, W_s, h_t, W_t, mask=None, T: float = 1.0, chunk: int = 0, loss=None,
                       grad_h=None, grad_W=None, workspace=None, err_flags=None, stream=None):
    """Full-vocabulary (K = V) distillation loss with the teacher computed in the
    same pass (see include/kd_full_kl.h).  bf16 inputs.  Returns (loss [1],
    grad_h [N, d_s], grad_W [V, d_s], workspace); asynchronous."""
    import torch
    for name, t in (("h_s", h_s), ("W_s", W_s), ("h_t", h_t), ("W_t", W_t)):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be a contiguous bfloat16 CUDA tensor")
    N, d_s = h_s.shape
    V, d_s2 = W_s.shape
    N2, d_t = h_t.shape
    V2, d_t2 = W_t.shape
    if d_s2 != d_s or d_t2 != d_t or N2 != N or V2 != V:
        raise ValueError("shape mismatch")
    if mask is not None and (mask.dtype != torch.uint8 or not mask.is_cuda
                             or not mask.is_contiguous() or mask.shape != (N,)):
        raise TypeError("mask must be a contiguous uint8 CUDA tensor of shape [N]")
    dev = h_s.device
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=dev)
    if grad_h is None:
        grad_h = torch.empty((N, d_s), dtype=torch.float32, device=dev)
    if grad_W is None:
        grad_W = torch.empty((V, d_s), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(full_kl_workspace_bytes(N, d_s, d_t, V, chunk), dtype=torch.uint8,
                                device=dev)
    st = load_library().kd_full_kl_fwd_bwd(
        _ptr(h_s), _ptr(W_s), _ptr(h_t), _ptr(W_t), _ptr(mask), N, d_s, d_t, V, float(T),
        int(chunk), _ptr(loss), _ptr(grad_h), _ptr(grad_W), _ptr(workspace), workspace.numel(),
        _ptr(err_flags), _stream_handle(stream))
    _check(st, "kd_full_kl_fwd_bwd")
    return loss, grad_h, grad_W, workspace


def kd_umma_gemm_bf16(A, B, M: int, N: int, K: int, a_mn_major: bool, b_mn_major: bool,
                      out=None, accumulate: bool = False, err_flags=None, stream=None):
    """D[M, N] (+)= A(m, k) B(n, k) on the tensor cores (see kd_topk_kl_steps.h)."""
    import torch
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    counter = torch.empty(1, dtype=torch.int32, device=A.device)
    if err_flags is None:
        err_flags = torch.zeros(1, dtype=torch.int32, device=A.device)
    st = load_library().kd_umma_gemm_bf16(_ptr(A), _ptr(B), _ptr(out), M, N, K, int(a_mn_major),
                                          int(b_mn_major), int(accumulate), _ptr(counter),
                                          _ptr(err_flags), _stream_handle(stream))
    _check(st, "kd_umma_gemm_bf16")
    return out, err_flags


def kd_timing_enable(on: bool = True):
    """Bracket every kernel launch of the library with CUDA events (see
    kd_topk_kl_steps.h)."""
    _check(load_library().kd_timing_enable(int(on)), "kd_timing_enable")


def kd_timing_collect():
    """Waits for the recorded events; returns {kernel kind: (launches, total ms)}
    and clears the record."""
    arr = (TimingEntry * 32)()
    n = ctypes.c_int32(0)
    _check(load_library().kd_timing_collect(arr, 32, ctypes.byref(n)), "kd_timing_collect")
    return {arr[i].name.decode(): (int(arr[i].launches), float(arr[i].total_ms))
            for i in range(min(n.value, 32))}


def kd_topk_kl_prepare(topk_idx, topk_logit, mask, N: int, d: int, V: int, T: float = 1.0,
                       chunk: int = 0, dtype: int = KD_BF16, workspace=None, n_valid=None,
                       err_flags=None, stream=None):
    """Teacher preparation and the valid-row count of this rank's tokens, the
    first half of a data-parallel step (see include/kd_topk_kl.h).  Returns
    (n_valid [1] int64 on the device, workspace)."""
    import torch
    for name, t in (("topk_idx", topk_idx), ("topk_logit", topk_logit)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if topk_idx.dtype != torch.int32 or topk_logit.dtype != torch.float32:
        raise TypeError("topk_idx must be int32 and topk_logit float32")
    if topk_idx.shape != topk_logit.shape or topk_idx.shape[0] != N:
        raise ValueError("shape mismatch")
    if mask is not None and (mask.dtype != torch.uint8 or not mask.is_cuda
                             or not mask.is_contiguous() or mask.shape != (N,)):
        raise TypeError("mask must be a contiguous uint8 CUDA tensor of shape [N]")
    K = topk_idx.shape[1]
    dev = topk_idx.device
    if workspace is None:
        workspace = allocate_workspace(N, d, V, K, chunk, dtype, dev)
    if n_valid is None:
        n_valid = torch.empty(1, dtype=torch.int64, device=dev)
    st = load_library().kd_topk_kl_prepare(
        _ptr(topk_idx), _ptr(topk_logit), _ptr(mask), N, d, V, K, float(T), int(chunk), dtype,
        _ptr(workspace), workspace.numel(), _ptr(n_valid), _ptr(err_flags), _stream_handle(stream))
    _check(st, "kd_topk_kl_prepare")
    return n_valid, workspace


def kd_topk_kl_fwd_bwd_prepared(h, W, K: int, workspace, n_norm=None, T: float = 1.0,
                                chunk: int = 0, loss=None, grad_h=None, grad_W=None,
                                err_flags=None, stream=None):
    """The chunk loop over a workspace that kd_topk_kl_prepare filled, with the
    loss divided by n_norm ([1] int64 on the device; None: this rank's own
    count).  Returns (loss, grad_h, grad_W)."""
    import torch
    for name, t in (("h", h), ("W", W)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if h.dtype != W.dtype:
        raise TypeError("h and W must have the same dtype")
    if n_norm is not None and (n_norm.dtype != torch.int64 or n_norm.device != h.device):
        raise TypeError("n_norm must be an int64 tensor on h's device")
    N, d = h.shape
    V = W.shape[0]
    dt = _dtype_code(h)
    dev = h.device
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=dev)
    if grad_h is None:
        grad_h = torch.empty((N, d), dtype=torch.float32, device=dev)
    if grad_W is None:
        grad_W = torch.empty((V, d), dtype=torch.float32, device=dev)
    st = load_library().kd_topk_kl_fwd_bwd_prepared(
        _ptr(h), _ptr(W), dt, N, d, V, int(K), float(T), int(chunk), _ptr(n_norm), _ptr(loss),
        _ptr(grad_h), _ptr(grad_W), _ptr(workspace), workspace.numel(), _ptr(err_flags),
        _stream_handle(stream))
    _check(st, "kd_topk_kl_fwd_bwd_prepared")
    return loss, grad_h, grad_W


def kd_topk_kl_fwd_prepared(h, W, K: int, workspace, n_norm=None, T: float = 1.0,
                            chunk: int = 0, loss=None, err_flags=None, stream=None):
    """The loss alone over a prepared workspace, divided by n_norm.  Returns loss."""
    import torch
    if h.dtype != W.dtype:
        raise TypeError("h and W must have the same dtype")
    N, d = h.shape
    V = W.shape[0]
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=h.device)
    st = load_library().kd_topk_kl_fwd_prepared(
        _ptr(h), _ptr(W), _dtype_code(h), N, d, V, int(K), float(T), int(chunk), _ptr(n_norm),
        _ptr(loss), _ptr(workspace), workspace.numel(), _ptr(err_flags), _stream_handle(stream))
    _check(st, "kd_topk_kl_fwd_prepared")
    return loss


def fwd_bwd_dp(h, W, topk_idx, topk_logit, mask=None, T: float = 1.0, chunk: int = 0,
               group=None, loss=None, grad_h=None, grad_W=None, workspace=None, err_flags=None,
               stream=None):
    """One data-parallel step of the loss over this rank's token shard.

    The batch's loss is the mean over all its valid tokens, so every rank
    divides by the batch's N_valid: prepare this shard (its count on the
    device), all-reduce the count, run the chunk loop with that divisor, then
    all-reduce loss and grad_W (the reduction a data-parallel training loop
    performs on its gradients anyway).  Every collective runs on the current
    stream; nothing waits on the host.  grad_h rows stay with their rank.
    With one rank (or torch.distributed not initialised) no collective runs
    and the result equals kd_topk_kl_fwd_bwd.

    Returns (loss [1], grad_h [N_r, d], grad_W [V, d], n_valid_total [1] int64,
    workspace)."""
    import torch.distributed as dist
    N, d, V, K = _validate(h, W, topk_idx, topk_logit, mask)
    dt = _dtype_code(h)
    world = dist.get_world_size(group) if dist.is_available() and dist.is_initialized() else 1
    n_valid, workspace = kd_topk_kl_prepare(topk_idx, topk_logit, mask, N, d, V, T, chunk, dt,
                                            workspace=workspace, err_flags=err_flags,
                                            stream=stream)
    if world > 1:
        dist.all_reduce(n_valid, group=group)
    loss, grad_h, grad_W = kd_topk_kl_fwd_bwd_prepared(
        h, W, K, workspace, n_norm=n_valid, T=T, chunk=chunk, loss=loss, grad_h=grad_h,
        grad_W=grad_W, err_flags=err_flags, stream=stream)
    if world > 1:
        dist.all_reduce(grad_W, group=group)
        dist.all_reduce(loss, group=group)
    return loss, grad_h, grad_W, n_valid, workspace


def status_string(st: int) -> str:
    return load_library().kd_status_string(st).decode()


def workspace_view(workspace, lay: WorkspaceLayout, name: str, count: int, dtype):
    """A typed view of the first `count` elements of one documented region of a
    workspace (see kd_topk_kl_workspace_layout), e.g. 'rows', 'lse',
    'idx_sorted', 'p_sorted', 'plogp', 'boff' or 'g'."""
    import torch
    off = getattr(lay, "off_" + name)
    nbytes = count * torch.empty(0, dtype=dtype).element_size()
    return workspace[off: off + nbytes].view(dtype)


# Short names.
fwd_bwd = kd_topk_kl_fwd_bwd
fwd = kd_topk_kl_fwd
fwd_bwd_noalloc = kd_topk_kl_fwd_bwd_noalloc
prepare = kd_topk_kl_prepare
fwd_bwd_prepared = kd_topk_kl_fwd_bwd_prepared
fwd_prepared = kd_topk_kl_fwd_prepared
topk_cache_build = kd_topk_cache_build
full_kl_fwd_bwd = kd_full_kl_fwd_bwd
timing_enable = kd_timing_enable
timing_collect = kd_timing_collect
