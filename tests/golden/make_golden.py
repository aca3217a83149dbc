"""Writes oracle_snapshot_small.json: the fp64 oracle's outputs on one small seeded problem.

Calls only the oracle and the seeded input generator. Rerun it (and say why in the
commit message, naming the passage of the LAGA page that justifies the change) only
when the oracle's arithmetic is deliberately changed.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from mla_attention_sequence_gb300.configs import Problem  # noqa: E402
from mla_attention_sequence_gb300.synth import make_inputs  # noqa: E402

PROBLEM = dict(B=1, Sq=4, S=7, n_h=2, d_c=5, d_nope=3, d_rope=2, d_v=3, q_offset=3, causal=True,
               dtype="f32")
SEED = 4242


def main():
    p = Problem(**PROBLEM)
    x = {k: v.astype(np.float64) for k, v in make_inputs(p, SEED).items()}
    out, lse = oracle.mla_forward(x["q"], x["c_kv"], x["k_rope"], x["W_UK"], x["W_UV"],
                                  p.q_offset, p.causal)
    g = oracle.mla_backward(x["q"], x["c_kv"], x["k_rope"], x["W_UK"], x["W_UV"], x["dout"],
                            p.q_offset, p.causal)
    snap = {
        "source": "fp64 oracle of the explicit MLA form (LAGA page, Abstract); written by "
                  "tests/golden/make_golden.py",
        "problem": PROBLEM, "seed": SEED,
        "out": out.tolist(), "lse": lse.tolist(),
        **{k: v.tolist() for k, v in g.items()},
    }
    with open(os.path.join(HERE, "oracle_snapshot_small.json"), "w") as f:
        json.dump(snap, f, indent=None)
        f.write("\n")


if __name__ == "__main__":
    main()
