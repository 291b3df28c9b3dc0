"""Stored expected values under tests/golden/ still match what produced them.

``tiny_fp16_noncausal_oracle.json`` was written by ``make_golden.py`` from the
fp64 oracle; a change to the oracle's arithmetic shows up here first.
``pages_values.json`` holds figures the pages print (with their citation);
the package's host-side helpers must reproduce them.
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


def test_pages_score_matrix_figures():
    from exact_attention_forward_10_gb300 import layer
    with open(os.path.join(HERE, "pages_values.json")) as f:
        g = json.load(f)["score_matrix"]
    assert layer.score_matrix_bytes(1, 1, g["T"], g["dtype_bytes"]) == g["bytes_per_head"]
    assert layer.score_matrix_bytes(g["B"], g["H"], g["T"], g["dtype_bytes"]) == g["bytes_per_batch"]
