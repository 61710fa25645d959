"""Writes oracle_tiny.json: the fp64 oracle's outputs on one tiny seeded case.

The pages print no worked example, so this file is not a page value: it is a
regression record that only this script writes, from ``oracle/`` alone, so that
any later change to the oracle's arithmetic shows up as a diff.  Run it from
the repository root:  python tests/golden/make_oracle_fixture.py
"""
import json
import math
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from exact_attention_98_gb300.inputs import attention_inputs  # noqa: E402

B, H, N, D, SEED = 1, 1, 16, 8, 0


def main():
    q, k, v, do = (t.double().numpy()[0, 0] for t in attention_inputs(B, H, N, D, seed=SEED))
    scale = 1.0 / math.sqrt(D)
    out = {"shape": [B, H, N, D], "seed": SEED, "scale": scale, "cases": {}}
    for causal in (False, True):
        o, lse = oracle.fwd_head(q, k, v, scale, causal)
        dq, dk, dv = oracle.bwd_head(q, k, v, do, scale, causal)
        out["cases"]["causal" if causal else "full"] = {
            "o": o.tolist(), "lse": lse.tolist(), "dq": dq.tolist(), "dk": dk.tolist(), "dv": dv.tolist()}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_tiny.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=0)


if __name__ == "__main__":
    main()
