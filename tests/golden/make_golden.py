"""Writes kda_exact_tiny.json: exact rational KDA results for a few tiny inputs.

Calls only ``oracle.exact`` (the Fraction brute force of the Kimi K3 --
Architecture Notes, section 1.1 recurrence). Run from the repository root:
``python tests/golden/make_golden.py``.
"""
import json
import os
import sys
from fractions import Fraction

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
from oracle.exact import kda_exact  # noqa: E402


def case(T, dk, dv, seed):
    # a small linear congruential sequence keeps the fixture independent of any RNG library
    state = seed

    def nxt(lo, hi, den):
        nonlocal state
        state = (state * 1103515245 + 12345) % (1 << 31)
        return Fraction(lo * den + state % ((hi - lo) * den + 1), den)

    q = [[nxt(-1, 1, 8) for _ in range(dk)] for _ in range(T)]
    k = [[nxt(-1, 1, 8) for _ in range(dk)] for _ in range(T)]
    v = [[nxt(-2, 2, 4) for _ in range(dv)] for _ in range(T)]
    alpha = [[nxt(0, 1, 8) * Fraction(7, 8) + Fraction(1, 8) for _ in range(dk)] for _ in range(T)]  # in [1/8, 1]
    beta = [nxt(0, 1, 8) for _ in range(T)]
    S0 = [[nxt(-1, 1, 4) for _ in range(dv)] for _ in range(dk)]
    o, S = kda_exact(q, k, v, alpha, beta, S0)
    s = lambda m: [[str(x) for x in r] for r in m]
    return {"q": s(q), "k": s(k), "v": s(v), "alpha": s(alpha), "beta": [str(b) for b in beta],
            "S0": s(S0), "o": s(o), "S_T": s(S)}


if __name__ == "__main__":
    out = {"source": "exact rational brute force (oracle.exact) of Kimi K3 -- Architecture Notes, "
                     "section 1.1: S_t = (I - b k k^T) Diag(a) S_{t-1} + b k v^T, o_t = S_t^T q_t",
           "cases": [case(4, 2, 3, 1), case(5, 3, 2, 2), case(3, 3, 3, 3)]}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "kda_exact_tiny.json")
    with open(path, "w") as fh:
        json.dump(out, fh, indent=1)
    print("wrote", path)
