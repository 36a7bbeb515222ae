"""Writes tests/golden/oracle_small.json from the fp64 oracle alone.

The pages print no worked numeric example of the attention backward pass
(the forward/backward tables in "[Issue]: Backward performance" and the
timings in triton #1806 are times, not values), so this fixture is a
regression record of the oracle itself, on small hand-chosen inputs: it
catches any later, unintended change to the oracle's arithmetic.  Inputs are
fixed rationals written here, not drawn from any generator.

Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
from oracle import attn_ref  # noqa: E402


def inputs():
    # B=1, Hq=2, Hkv=1, Nq=Nkv=3, d=2: small rationals with distinct rows.
    q = np.array([[[[0.5, -1.0], [1.25, 0.75], [-0.5, 0.25]],
                   [[1.0, 0.5], [-0.25, -0.75], [0.0, 1.5]]]])
    k = np.array([[[[0.25, 1.0], [-1.0, 0.5], [0.75, -0.25]]]])
    v = np.array([[[[1.0, -2.0], [0.5, 0.25], [-1.5, 1.0]]]])
    do = np.array([[[[0.125, 1.0], [-0.5, 0.5], [1.0, -0.25]],
                    [[-1.0, 0.375], [0.25, 0.25], [0.5, -1.5]]]])
    return q, k, v, do


def main():
    q, k, v, do = inputs()
    out = {"note": "oracle regression record; inputs are fixed rationals (see make_golden.py)",
           "q": q.tolist(), "k": k.tolist(), "v": v.tolist(), "do": do.tolist(), "cases": []}
    for causal in (False, True):
        for scale in (1.0, 0.7):
            o, lse = attn_ref.forward(q, k, v, scale, causal)
            g = attn_ref.backward(q, k, v, do, scale, causal)
            out["cases"].append({"causal": causal, "scale": scale, "o": o.tolist(), "lse": lse.tolist(),
                                 "dq": g["dq"].tolist(), "dk": g["dk"].tolist(), "dv": g["dv"].tolist(),
                                 "D": g["D"].tolist()})
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
