"""The oracle still reproduces its committed snapshot (tests/golden/oracle_snapshot_small.json)."""
import json
import os

import numpy as np

import oracle
from mla_attention_sequence_gb300.configs import Problem
from mla_attention_sequence_gb300.synth import make_inputs

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_matches_snapshot():
    with open(os.path.join(HERE, "golden", "oracle_snapshot_small.json")) as f:
        snap = json.load(f)
    p = Problem(**snap["problem"])
    x = {k: v.astype(np.float64) for k, v in make_inputs(p, snap["seed"]).items()}
    out, lse = oracle.mla_forward(x["q"], x["c_kv"], x["k_rope"], x["W_UK"], x["W_UV"],
                                  p.q_offset, p.causal)
    g = oracle.mla_backward(x["q"], x["c_kv"], x["k_rope"], x["W_UK"], x["W_UV"], x["dout"],
                            p.q_offset, p.causal)
    np.testing.assert_allclose(out, snap["out"], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse, snap["lse"], rtol=1e-13, atol=1e-15)
    for k in ("dq", "dc_kv", "dk_rope", "dW_UK", "dW_UV"):
        np.testing.assert_allclose(g[k], snap[k], rtol=1e-12, atol=1e-14)
