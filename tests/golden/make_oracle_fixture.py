"""Writes ``oracle_gqa_b1_t7.txt`` and ``oracle_varlen_tq_tk.txt``: the fp64
oracle's outputs on one small fixed-length grouped-query case and one packed
variable-length case with Tq != Tk, both with exactly representable inputs.

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


# A packed variable-length case with Tq != Tk: more queries than keys (rows
# that see no key under the causal mask), fewer, and a sequence with no keys.
VARLEN_TQ, VARLEN_TK = [5, 2, 4, 3], [3, 6, 4, 0]
VARLEN_NAME = "oracle_varlen_tq_tk.txt"


def varlen_inputs():
    """Packed Q, K, V, dO with entries in {-1, -7/8, ..., 1}."""
    nq, nk = sum(VARLEN_TQ), sum(VARLEN_TK)

    def pattern(rows, H, salt):
        x = np.empty((rows, H, D))
        for t in range(rows):
            for h in range(H):
                for d in range(D):
                    x[t, h, d] = ((t * 5 + h * 7 + d * 3 + salt) % 17 - 8) / 8.0
        return x
    return pattern(nq, HQ, 1), pattern(nk, HKV, 6), pattern(nk, HKV, 11), pattern(nq, HQ, 2)


def varlen_outputs(causal):
    q, k, v, do = varlen_inputs()
    cu_q = np.concatenate([[0], np.cumsum(VARLEN_TQ)])
    cu_k = np.concatenate([[0], np.cumsum(VARLEN_TK)])
    o, lse = oracle.attn_fwd_varlen(q, k, v, cu_q, cu_k, SCALE, causal)
    dq, dk, dv, _, _ = oracle.attn_bwd_varlen(q, k, v, do, cu_q, cu_k, SCALE, causal)
    return {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}


def _write(name, header, outputs_of):
    lines = header
    for causal in (1, 0):
        for tensor, x in outputs_of(bool(causal)).items():
            vals = " ".join(f"{v:.17g}" for v in x.reshape(-1))
            lines.append(f"causal={causal} {tensor} {vals}")
    with open(os.path.join(HERE, name), "w") as f:
        f.write("\n".join(lines) + "\n")


def main():
    _write(NAME, [f"# fp64 oracle, B={B} T={T} Hq={HQ} Hkv={HKV} D={D} scale={SCALE}; inputs from",
                  "# make_oracle_fixture.inputs(); one line per tensor, row-major, 17 significant "
                  "digits"],
           outputs)
    _write(VARLEN_NAME,
           [f"# fp64 oracle, packed varlen: tq={VARLEN_TQ} tk={VARLEN_TK} Hq={HQ} Hkv={HKV} D={D} "
            f"scale={SCALE}; inputs from",
            "# make_oracle_fixture.varlen_inputs(); one line per tensor, row-major, 17 significant "
            "digits (-inf: LSE of a row that sees no key)"],
           varlen_outputs)


if __name__ == "__main__":
    main()
