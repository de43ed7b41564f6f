"""Seeded synthetic inputs for the top-K KL distillation loss.

This module only draws numbers: the student hidden states h[N,d], the LM-head
weight W[V,d], the teacher top-K cache (int32 index, fp32 logit) and the token
mask. It holds none of the loss's arithmetic, so both the fp64 oracle and the
CUDA path can take their inputs from here without sharing any of the method.

Workload shapes follow the write-ups of "Efficient Knowledge Distillation for
LLMs: Offline Top-K Logits and a Fused Chunked KL Loss": a teacher cache of the
top 100 entries per position (ai2day.live story, "What did the researchers
change?"), a gpt-oss-120b-sized vocabulary of 201,088 at 32K context with
batch 4 ("Why is this so hard to do cheaply?") and a Llama-3.1-8B -> 3.2B
student (aiphreaks.com summary).

Recipe (numpy PCG64 Generator seeded with `seed`, drawing in this order:
h, W, idx, logit noise, head gap; the mask comes from its own PCG64 stream
seeded with [mask_seed, 1], mask_seed = seed + 100 j for the first j >= 0
whose masked fraction falls in mask_frac_range when one is given):
  * h ~ N(0, h_std^2), W ~ N(0, w_std^2), drawn fp32; bf16 configs round them
    to bf16 with round-to-nearest-even.
  * idx: K distinct values per row, uniform in [0, V): draw 2K candidates, keep
    the first K distinct ones in draw order, redraw the rare row that has fewer
    (when 4K > V: the first K entries of a random permutation instead).
  * teacher logits: base - 2 ln k + N(0, 0.5^2) for k = 1..K, sorted descending
    (index position k pairs with the k-th largest value).  The heavy-head
    variant draws the tail l_2..l_K that way and sets l_1 = l_2 + Exp(rate 2).
  * packed mask: each sequence is filled with documents of length U[doc_lo,
    doc_hi] (mask 1), each followed by a padding run of length U[pad_lo,
    pad_hi] (mask 0); a run cut by the end of the sequence is kept.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even).

    Returns the 16-bit patterns as uint16.  Inputs here are finite."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class KDInputs:
    """One synthetic problem.  For dtype 'bf16', h and W hold uint16 bf16 bit
    patterns; for 'fp32' they hold float32 values."""
    name: str
    dtype: str
    h: np.ndarray
    W: np.ndarray
    idx: np.ndarray
    logit: np.ndarray
    mask: Optional[np.ndarray]
    T: float
    seed: int

    @property
    def N(self) -> int:
        return int(self.h.shape[0])

    @property
    def d(self) -> int:
        return int(self.h.shape[1])

    @property
    def V(self) -> int:
        return int(self.W.shape[0])

    @property
    def K(self) -> int:
        return int(self.idx.shape[1])

    def h_f32(self) -> np.ndarray:
        return bf16_bits_to_f32(self.h) if self.dtype == "bf16" else self.h

    def W_f32(self) -> np.ndarray:
        return bf16_bits_to_f32(self.W) if self.dtype == "bf16" else self.W

    def masked_fraction(self) -> float:
        if self.mask is None:
            return 0.0
        return float(1.0 - self.mask.mean())


def distinct_indices(rng: np.random.Generator, N: int, K: int, V: int) -> np.ndarray:
    """K distinct uniform indices in [0, V) per row, first-K-distinct in draw order."""
    if K > V:
        raise ValueError("cannot draw K distinct indices from fewer than K values")
    out = np.empty((N, K), dtype=np.int32)
    if 4 * K > V:
        # dense case: the first K entries of a random permutation of [0, V)
        keys = rng.random((N, V))
        return np.argsort(keys, axis=1)[:, :K].astype(np.int32)
    todo = np.arange(N)
    while todo.size:
        n = todo.size
        width = max(2 * K, K + 8)
        cand = rng.integers(0, V, size=(n, width), dtype=np.int64)
        order = np.argsort(cand, axis=1, kind="stable")
        srt = np.take_along_axis(cand, order, axis=1)
        dup_sorted = np.zeros_like(srt, dtype=bool)
        dup_sorted[:, 1:] = srt[:, 1:] == srt[:, :-1]
        dup = np.empty_like(dup_sorted)
        np.put_along_axis(dup, order, dup_sorted, axis=1)
        keep = ~dup
        rank = np.cumsum(keep, axis=1)
        ok = rank[:, -1] >= K
        sel = keep & (rank <= K)
        rows_ok = np.nonzero(ok)[0]
        if rows_ok.size:
            vals = cand[rows_ok][sel[rows_ok]].reshape(rows_ok.size, K)
            out[todo[rows_ok]] = vals.astype(np.int32)
        todo = todo[~ok]
    return out


def teacher_logits(rng: np.random.Generator, N: int, K: int, base: float,
                   heavy_head: bool) -> np.ndarray:
    k = np.arange(1, K + 1, dtype=np.float64)
    noise = rng.normal(0.0, 0.5, size=(N, K))
    vals = base - 2.0 * np.log(k)[None, :] + noise
    vals = -np.sort(-vals, axis=1)
    if heavy_head:
        gap = rng.exponential(scale=0.5, size=N)  # rate 2
        tail = vals[:, : K - 1] if K > 1 else vals[:, :0]
        head = (tail[:, 0] if K > 1 else vals[:, 0]) + gap
        vals = np.concatenate([head[:, None], tail], axis=1)
    return vals.astype(np.float32)


def packed_mask(rng: np.random.Generator, B: int, S: int, doc=(1200, 3550),
                pad=(16, 512)) -> np.ndarray:
    m = np.zeros((B, S), dtype=np.uint8)
    for b in range(B):
        pos = 0
        while pos < S:
            n = int(rng.integers(doc[0], doc[1] + 1))
            m[b, pos: pos + n] = 1
            pos += n
            pos += int(rng.integers(pad[0], pad[1] + 1))
    return m.reshape(-1)


def make_inputs(N: int, d: int, V: int, K: int, *, T: float = 1.0, dtype: str = "bf16",
                seed: int = 0, h_std: float = 1.0, w_std: float = 0.02,
                logit_base: float = 12.0, heavy_head: bool = False,
                mask: Optional[str] = None, B: int = 1, doc=(1200, 3550), pad=(16, 512),
                mask_frac_range=None, name: str = "custom") -> KDInputs:
    """Draw one problem.  mask is None, 'packed' (B sequences of N/B tokens) or
    'random<p>' (each token masked independently with probability p)."""
    if dtype not in ("bf16", "fp32"):
        raise ValueError(dtype)
    rng = np.random.Generator(np.random.PCG64(seed))
    h = rng.standard_normal((N, d), dtype=np.float32)
    if h_std != 1.0:
        h *= np.float32(h_std)
    W = rng.standard_normal((V, d), dtype=np.float32)
    W *= np.float32(w_std)
    idx = distinct_indices(rng, N, K, V)
    logit = teacher_logits(rng, N, K, logit_base, heavy_head)
    m = None
    mask_seed = seed
    for attempt in range(1000):
        mrng = np.random.Generator(np.random.PCG64([mask_seed, 1]))
        if mask == "packed":
            assert N % B == 0
            m = packed_mask(mrng, B, N // B, doc, pad)
        elif mask is not None and mask.startswith("random"):
            prob = float(mask[len("random"):])
            m = (mrng.random(N) >= prob).astype(np.uint8)
        if m is None or mask_frac_range is None:
            break
        frac = 1.0 - m.mean()
        if mask_frac_range[0] <= frac <= mask_frac_range[1]:
            break
        mask_seed += 100
    else:
        raise RuntimeError("no mask seed gives the requested masked fraction")
    if dtype == "bf16":
        h = bf16_bits(h)
        W = bf16_bits(W)
    return KDInputs(name=name, dtype=dtype, h=h, W=W, idx=idx, logit=logit, mask=m,
                    T=float(T), seed=seed)


# The five workloads: a tiny fp32 case, a Llama-style 3B student, the
# large-vocabulary 32K-token case, the same batched to 128K tokens, and a
# packed/masked case with temperature 2.
CONFIGS = {
    1: dict(name="tiny-fp32", N=64, d=64, V=512, K=8, T=1.0, dtype="fp32", seed=0,
            h_std=1.0, w_std=float(1.0 / np.sqrt(64)), logit_base=8.0),
    2: dict(name="llama3b-8k", N=8192, d=3072, V=128256, K=100, T=1.0, dtype="bf16",
            seed=1),
    3: dict(name="vocab201k-32k", N=32768, d=2880, V=201088, K=100, T=1.0, dtype="bf16",
            seed=2),
    4: dict(name="vocab201k-128k", N=131072, d=2880, V=201088, K=100, T=1.0,
            dtype="bf16", seed=3),
    5: dict(name="packed-masked-T2", N=32768, d=4096, V=151936, K=100, T=2.0,
            dtype="bf16", seed=4, heavy_head=True, mask="packed", B=2,
            mask_frac_range=(0.08, 0.12)),
}


def make_config(i: int, **overrides) -> KDInputs:
    """Config i (1..5).  Keyword overrides (N, V, d, doc, pad, ...) give smaller
    problems of the same kind; a packed mask with a smaller N keeps the masked
    fraction near 10% only if doc and pad are scaled with it."""
    c = dict(CONFIGS[i])
    c.update(overrides)
    return make_inputs(**c)


def full_teacher_config(c: dict) -> dict:
    """The teacher of a full-vocabulary workload built from the student's
    recipe c: the same sizes (so d_t = d_s), its own seed, no mask; its top-K
    fields are unused (K = 1)."""
    ct = dict(c)
    ct["seed"] = c["seed"] + 50
    ct["mask"] = None
    ct.pop("mask_frac_range", None)
    ct["K"] = 1
    return ct


def make_full_teacher_pair(i: int, **overrides):
    """(student, teacher) inputs of the full-vocabulary workload on config i:
    the student is config i (with the overrides), the teacher
    full_teacher_config of it; both models' h and W are used."""
    c = dict(CONFIGS[i])
    c.update(overrides)
    return make_inputs(**c), make_inputs(**full_teacher_config(c))
