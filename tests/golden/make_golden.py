"""Writes the golden regression fixture for the tiny fp32 workload.

The write-ups print no worked numeric example, so the stored values come from
the fp64 oracle (and the seeded input generator) only, after the oracle's pins
in tests/test_oracle.py pass.  Run from the repository root:
    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from top_kl_loss_token_b300 import synth  # noqa: E402


def main():
    x = synth.make_config(1)
    r = oracle.fwd_bwd(x.h_f32(), x.W_f32(), x.idx, x.logit, x.mask, x.T)
    out = dict(
        workload="tiny fp32: N=64, d=64, V=512, K=8, T=1, seed 0",
        loss=r["loss"],
        grad_h_abs_sum=float(np.abs(r["grad_h"]).sum()),
        grad_W_abs_sum=float(np.abs(r["grad_W"]).sum()),
        lse_first8=[float(v) for v in r["lse"][:8]],
    )
    with open(os.path.join(HERE, "config1_tiny_fp32.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
