"""Stored expected values under tests/golden/ still match what produced them.

``tiny_fp16_noncausal_oracle.json`` was written by ``make_golden.py`` from the
fp64 oracle; a change to the oracle's arithmetic shows up here first.
``pages_values.json`` holds the figures the pages print (with citations); the
package's host-side helpers must reproduce them.
"""
import json
import os

import numpy as np

import attn_inputs
import oracle

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_tiny_oracle_fixture():
    with open(os.path.join(HERE, "tiny_fp16_noncausal_oracle.json")) as f:
        g = json.load(f)
    w = attn_inputs.WORKLOADS["tiny"]
    x = w.inputs()
    o, lse = oracle.attn_fwd(x.q, x.k, x.v, False, w.scale)
    np.testing.assert_allclose(lse.reshape(-1), g["lse"], rtol=0, atol=1e-12)
    flat = o.reshape(-1, w.D)
    for r, vals in g["o_rows"].items():
        np.testing.assert_allclose(flat[int(r)], vals, rtol=0, atol=1e-12)
