"""Writes ``oracle_gqa_b1_t7.txt``: the fp64 oracle's outputs on one small
grouped-query case with exactly representable inputs.

The pages print no worked attention example (no inputs with their outputs),
so no stored value here comes from them.  This fixture is a regression anchor
for the oracle alone: it is written by this script, which calls only the
oracle, and ``test_oracle.py`` checks that the oracle still reproduces it.  A
change to the oracle's arithmetic that moves these numbers has to be argued
from the pages' definitions, not from this file.

Run from the repository root:  python tests/golden/make_oracle_fixture.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402

B, T, HQ, HKV, D = 1, 7, 4, 2, 3
SCALE = 0.5
NAME = "oracle_gqa_b1_t7.txt"


def inputs():
    """Q, K, V, dO with entries in {-1, -7/8, ..., 1}: exact in bf16 and fp64."""
    def pattern(H, salt):
        x = np.empty((B, T, H, D))
        for t in range(T):
            for h in range(H):
                for d in range(D):
                    x[0, t, h, d] = ((t * 7 + h * 3 + d * 5 + salt) % 17 - 8) / 8.0
        return x
    return pattern(HQ, 0), pattern(HKV, 4), pattern(HKV, 9), pattern(HQ, 13)


def outputs(causal):
    q, k, v, do = inputs()
    o, lse = oracle.attn_fwd(q, k, v, SCALE, causal)
    dq, dk, dv, _, _ = oracle.attn_bwd(q, k, v, do, SCALE, causal)
    return {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}


def main():
    lines = [f"# fp64 oracle, B={B} T={T} Hq={HQ} Hkv={HKV} D={D} scale={SCALE}; inputs from",
             "# make_oracle_fixture.inputs(); one line per tensor, row-major, 17 significant digits"]
    for causal in (1, 0):
        for name, x in outputs(bool(causal)).items():
            vals = " ".join(f"{v:.17g}" for v in x.reshape(-1))
            lines.append(f"causal={causal} {name} {vals}")
    with open(os.path.join(HERE, NAME), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
