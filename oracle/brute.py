"""Pure-Python decode attention for tiny inputs — TEST INFRASTRUCTURE ONLY.

Scalar loops with ``math.fsum`` (exactly rounded sums) and ``math.exp``: the
textbook softmax(q . k / sqrt(D)) . v written out term by term, used to pin the
numpy oracle (attention.py) on inputs small enough to loop over.
"""
from __future__ import annotations

import math


def attend_brute(q_rows, k_rows, v_rows, sm_scale):
    """q_rows: G lists of D floats; k_rows / v_rows: L lists of D floats.

    Returns (out: G lists of D floats, lse: G floats)."""
    outs, lses = [], []
    L = len(k_rows)
    for q in q_rows:
        D = len(q)
        if L == 0:
            outs.append([0.0] * D)
            lses.append(-math.inf)
            continue
        z = [sm_scale * math.fsum(q[d] * k[d] for d in range(D)) for k in k_rows]
        m = max(z)
        e = [math.exp(zt - m) for zt in z]
        l = math.fsum(e)
        outs.append([math.fsum(e[t] * v_rows[t][d] for t in range(L)) / l for d in range(D)])
        lses.append(m + math.log(l))
    return outs, lses
