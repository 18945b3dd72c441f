"""Write tests/golden/small_case.json from the oracle alone.

The file pins the oracle against accidental change: it holds a small seeded
case (bf16-representable inputs, widened exactly) and the oracle's f64
outputs. Its forward is in turn pinned by the decimal brute force in
tests/oracle_checks.py. Regenerate only when a change to the oracle's
arithmetic is justified by the pages (and say which passage in the commit).

    python tests/golden/make_golden.py
"""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from gqa_inputs import make_inputs, to_f64  # noqa: E402

B, Hq, Hkv, S, D, SEED = 1, 4, 2, 7, 4, 5
CAUSAL, SCALE = True, 0.5


def main():
    q, k, v, dO = make_inputs(B, Hq, Hkv, S, D, SEED, do_std=1.0)
    q, k, v, dO = (to_f64(t) for t in (q, k, v, dO))
    O, L = oracle.forward(q, k, v, causal=CAUSAL, scale=SCALE)
    dQ, dK, dV = oracle.backward(q, k, v, dO, causal=CAUSAL, scale=SCALE)
    arrays = dict(q=q, k=k, v=v, dO=dO, O=O, LSE=L, dQ=dQ, dK=dK, dV=dV)
    out = {
        "meta": {"B": B, "Hq": Hq, "Hkv": Hkv, "S": S, "D": D, "seed": SEED,
                 "causal": CAUSAL, "scale": SCALE,
                 "written_by": "tests/golden/make_golden.py (oracle only)"},
        "arrays": {k_: a.tolist() for k_, a in arrays.items()},
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "small_case.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=None, separators=(",", ":"))
        f.write("\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
