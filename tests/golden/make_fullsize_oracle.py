"""Writes the fp64 oracle's results for the full-size workloads into a local
cache that the full-size GPU parity tests read.

At 32K and 128K tokens with a 201,088-word vocabulary the dense fp64 forward
takes minutes to tens of minutes of host time (2 N d V multiply-adds), too long
to repeat inside every test run, so it is computed once per input set and kept
in tests/.oracle_cache/ (not under version control: it is a few MB of binary
arrays and is rebuilt from the oracle and the seeded generator alone).

Every value stored here comes from oracle/ and the seeded input generator
(synth), never from the CUDA path.  Per workload:
  * the whole-batch loss, N_valid, and every token's lse and loss term (the
    oracle's full forward, rows processed in blocks);
  * about 2048 rows of grad_W (half the vocabulary rows of teacher entries of
    rank 1, half uniform, plus the first and the last row), each computed from
    the oracle's own lse.
For the full-vocabulary loss on config 3's sizes (student = config 3, teacher
drawn by synth.full_teacher_config, as the benchmark's --full-teacher mode
does): the whole-batch loss, every token's lse (of the student logits) and
loss term, and about 2048 grad_W rows (uniform vocabulary rows plus the first
and the last), from oracle/full_kl_oracle.py.
Each file carries a digest of the inputs it was computed from; a test that
finds a different digest recomputes.  A file whose grad_W rows are not the
current sample keeps its forward and recomputes those rows from its lse.

    python tests/golden/make_fullsize_oracle.py [config ...]  (default: 3 5 4 full3)
"""
import hashlib
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

CACHE_DIR = os.path.join(ROOT, "tests", ".oracle_cache")


def input_digest(x) -> str:
    """SHA-256 over the exact bits of one synthetic problem's inputs."""
    d = hashlib.sha256()
    for a in (x.h, x.W, x.idx, x.logit):
        d.update(np.ascontiguousarray(a).view(np.uint8).data)
    d.update(b"nomask" if x.mask is None else np.ascontiguousarray(x.mask).data)
    d.update(repr((x.dtype, x.T, x.N, x.d, x.V, x.K)).encode())
    return d.hexdigest()


def vocab_sample(x, n_teacher=1024, n_uniform=1024, seed=None) -> np.ndarray:
    """Vocabulary rows to check in grad_W: the rank-1 teacher index of
    n_teacher random tokens, n_uniform uniform rows, and rows 0 and V - 1."""
    rng = np.random.default_rng(1000 + x.seed if seed is None else seed)
    toks = rng.choice(x.N, size=min(n_teacher, x.N), replace=False)
    teach = x.idx[toks, 0].astype(np.int64)
    uni = rng.integers(0, x.V, size=n_uniform)
    return np.unique(np.concatenate([teach, uni, [0, x.V - 1]]))


def cache_path(cfg: int) -> str:
    return os.path.join(CACHE_DIR, f"config{cfg}.npz")


def compute(x, block_rows=512, log=None):
    """The oracle's whole-batch forward and sampled grad_W rows for x."""
    import oracle
    t0 = time.time()
    h = x.h_f32()
    W = x.W_f32()
    full = oracle.fwd(h, W, x.idx, x.logit, x.mask, x.T, block_rows=block_rows)
    t1 = time.time()
    vr = vocab_sample(x)
    gW = oracle.grad_W_rows(h, W, x.idx, x.logit, x.mask, x.T, vr, full["lse"])
    t2 = time.time()
    if log is not None:
        log(f"{x.name}: forward {t1 - t0:.0f} s, {vr.size} grad_W rows {t2 - t1:.0f} s")
    return dict(digest=np.array(input_digest(x)), loss=np.float64(full["loss"]),
                n_valid=np.int64(full["n_valid"]), lse=full["lse"],
                loss_rows=full["loss_rows"], vocab_rows=vr, grad_W_rows=gW)


def _save(path, res):
    os.makedirs(CACHE_DIR, exist_ok=True)
    tmp = path + f".tmp{os.getpid()}.npz"
    np.savez(tmp, **res)
    os.replace(tmp, path)


def _cached(path, digest):
    if not os.path.exists(path):
        return None
    with np.load(path) as z:
        if str(z["digest"]) != digest:
            return None
        return {k: z[k] for k in z.files}


def load_or_compute(cfg: int, x, log=None):
    """The cached oracle results for config cfg if they match x's inputs, else
    computed now (and cached)."""
    path = cache_path(cfg)
    res = _cached(path, input_digest(x))
    if res is None:
        res = compute(x, log=log)
        _save(path, res)
        return res
    vr = vocab_sample(x)
    if not np.array_equal(res["vocab_rows"], vr):
        # the same forward, another grad_W sample: those rows only
        import oracle
        res["vocab_rows"] = vr
        res["grad_W_rows"] = oracle.grad_W_rows(x.h_f32(), x.W_f32(), x.idx, x.logit, x.mask,
                                                x.T, vr, res["lse"])
        _save(path, res)
    return res


def full_vocab_sample(xs, n_uniform=2048) -> np.ndarray:
    """Vocabulary rows of grad_W checked for the full-vocabulary loss."""
    rng = np.random.default_rng(2000 + xs.seed)
    return np.unique(np.concatenate([rng.integers(0, xs.V, size=n_uniform), [0, xs.V - 1]]))


def full_cache_path(cfg: int) -> str:
    return os.path.join(CACHE_DIR, f"full_kl_config{cfg}.npz")


def compute_full(xs, xt, block_rows=256, log=None):
    """The full-vocabulary oracle's whole-batch forward and sampled grad_W
    rows for student xs and teacher xt."""
    import oracle
    t0 = time.time()
    hs, Ws, ht, Wt = xs.h_f32(), xs.W_f32(), xt.h_f32(), xt.W_f32()
    full = oracle.full_kl_fwd_bwd(hs, Ws, ht, Wt, xs.mask, xs.T, block_rows=block_rows,
                                  want_grads=False)
    t1 = time.time()
    vr = full_vocab_sample(xs)
    gW = oracle.full_kl_grad_W_rows(hs, Ws, ht, Wt, xs.mask, xs.T, vr, full["lse_s"],
                                    full["lse_t"])
    t2 = time.time()
    if log is not None:
        log(f"full-vocabulary {xs.name}: forward {t1 - t0:.0f} s, {vr.size} grad_W rows "
            f"{t2 - t1:.0f} s")
    return dict(digest=np.array(input_digest(xs) + input_digest(xt)),
                loss=np.float64(full["loss"]), n_valid=np.int64(full["n_valid"]),
                lse=full["lse_s"], lse_t=full["lse_t"], loss_rows=full["loss_rows"],
                vocab_rows=vr, grad_W_rows=gW)


def load_or_compute_full(cfg: int, xs, xt, log=None):
    """The cached full-vocabulary oracle results for config cfg if they match
    the inputs, else computed now (and cached)."""
    path = full_cache_path(cfg)
    res = _cached(path, input_digest(xs) + input_digest(xt))
    if res is None or "lse_t" not in res:
        res = compute_full(xs, xt, log=log)
        _save(path, res)
        return res
    vr = full_vocab_sample(xs)
    if not np.array_equal(res["vocab_rows"], vr):
        import oracle
        res["vocab_rows"] = vr
        res["grad_W_rows"] = oracle.full_kl_grad_W_rows(
            xs.h_f32(), xs.W_f32(), xt.h_f32(), xt.W_f32(), xs.mask, xs.T, vr, res["lse"],
            res["lse_t"])
        _save(path, res)
    return res


def main(argv):
    from top_kl_loss_token_b300 import synth
    args = list(argv) or ["3", "5", "4", "full3"]
    for a in args:
        if a.startswith("full"):
            cfg = int(a[4:])
            xs, xt = synth.make_full_teacher_pair(cfg)
            res = load_or_compute_full(cfg, xs, xt, log=lambda s: print(s, flush=True))
            print(f"full-vocabulary config {cfg}: loss {float(res['loss']):.9f}, N_valid "
                  f"{int(res['n_valid'])}, {res['vocab_rows'].size} grad_W rows -> "
                  f"{full_cache_path(cfg)}", flush=True)
            del xs, xt, res
            continue
        cfg = int(a)
        x = synth.make_config(cfg)
        res = load_or_compute(cfg, x, log=lambda s: print(s, flush=True))
        print(f"config {cfg}: loss {float(res['loss']):.9f}, N_valid {int(res['n_valid'])}, "
              f"{res['vocab_rows'].size} grad_W rows -> {cache_path(cfg)}", flush=True)
        del x, res


if __name__ == "__main__":
    main(sys.argv[1:])
