"""Writes tests/golden/*.json from the CPU oracle only (no GPU code is imported).

Run from the repository root:  python tests/golden/make_golden.py

Inputs are small, exactly representable (bf16-exact) values written out in this
script, so the fixture does not depend on any random number generator.
"""

import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402


def tiny_case():
    # B=1, H=1, N=5, d=2; every value has at most 8 significant bits.
    q = np.array([[0.5, -1.0], [1.25, 0.75], [-0.5, 2.0], [0.0, -0.25], [1.5, 1.5]])
    k = np.array([[1.0, 0.5], [-0.75, 0.25], [0.5, -1.5], [2.0, 0.0], [-1.0, -1.0]])
    v = np.array([[0.25, 1.0], [-2.0, 0.5], [1.0, -0.75], [0.125, 3.0], [-1.5, -0.5]])
    do = np.array([[1.0, -0.5], [0.25, 0.25], [-1.0, 2.0], [0.5, 0.0], [0.75, -1.25]])
    out = {"inputs": {"q": q.tolist(), "k": k.tolist(), "v": v.tolist(), "do": do.tolist()},
           "scale": 0.7071067811865476, "cases": {}}
    for causal in (False, True):
        args = [x[None, None] for x in (q, k, v)]
        o, lse = oracle.forward(*args, out["scale"], causal)
        dq, dk, dv = oracle.backward(*args, do[None, None], out["scale"], causal)
        out["cases"]["causal" if causal else "full"] = {
            "o": o[0, 0].tolist(), "lse": lse[0, 0].tolist(),
            "dq": dq[0, 0].tolist(), "dk": dk[0, 0].tolist(), "dv": dv[0, 0].tolist(),
        }
    return out


if __name__ == "__main__":
    with open(os.path.join(HERE, "tiny_n5_d2.json"), "w") as f:
        json.dump(tiny_case(), f, indent=1)
        f.write("\n")
