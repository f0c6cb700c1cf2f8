"""Writes the stored expected values under tests/golden/ (run from the repo root:
``python tests/golden/make_golden.py``).

It calls only the fp64 oracle (and the seeded input generators).  The pages
print no worked numeric example, so every stored value here is the oracle's:
the fixture guards against silent drift of the oracle and gives the GPU tests
a fixed anchor on the smallest workload (causal attention, B=1, H=2, L=256,
d=64, bf16 N(0,1) inputs from seed 0, scale 1/sqrt(d)).
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from flashattention_attn_fwd_gb300 import synth  # noqa: E402

ROWS = [(0, 0, 0), (0, 0, 1), (0, 0, 127), (0, 0, 128), (0, 1, 200), (0, 1, 255)]


def main():
    q, k, v = synth.attn_inputs(1, 2, 2, 256, 64, seed=0)
    out, lse = oracle.attention(q, k, v, mask="causal")
    fx = {
        "workload": "causal attention B=1 H=2 L=256 d=64, synth.attn_inputs seed 0",
        "rows": [list(r) for r in ROWS],
        "out": [[float(x) for x in out[b, h, i]] for (b, h, i) in ROWS],
        "lse": [float(lse[b, h, i]) for (b, h, i) in ROWS],
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "causal_b1h2l256d64_seed0.json")
    with open(path, "w") as f:
        json.dump(fx, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
