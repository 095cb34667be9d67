"""The oracle still reproduces the stored fixture written by tests/golden/make_golden.py."""

import json
import os

import numpy as np

import oracle

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_tiny_fixture_regression():
    with open(os.path.join(HERE, "tiny_n5_d2.json")) as f:
        g = json.load(f)
    q, k, v, do = (np.array(g["inputs"][n])[None, None] for n in ("q", "k", "v", "do"))
    for name, causal in (("full", False), ("causal", True)):
        ref = g["cases"][name]
        o, lse = oracle.forward(q, k, v, g["scale"], causal)
        dq, dk, dv = oracle.backward(q, k, v, do, g["scale"], causal)
        for got, key in ((o, "o"), (lse, "lse"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
            np.testing.assert_allclose(got[0, 0], np.array(ref[key]), rtol=1e-13, atol=1e-14)
