"""Brute-force attention in 50-digit arithmetic (mpmath), for tiny inputs.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  It uses the naive
softmax exp(s) / sum exp(s) with NO maximum subtracted ("Flash Attention 代码填空
(Level 2-3)", Exercise 2, naive_softmax): at 50 digits and with |s| far below
the exponent range this cannot overflow, and it shares no step with the
float64 oracle's max-subtracted passes, so agreement pins both.
"""
from __future__ import annotations

import numpy as np


def attention_mp(q, k, v, scale: float, digits: int = 50, limits=None):
    """Returns (O, LSE) as float64 arrays for one head: q [nq, d], k/v [nk, d].

    limits[i], if given, is the number of leading keys query row i may see.
    """
    import mpmath as mp

    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    nq, d = q.shape
    nk = k.shape[0]
    o = np.empty((nq, v.shape[1]))
    lse = np.empty(nq)
    with mp.workdps(digits):
        sc = mp.mpf(float(scale))
        kk = [[mp.mpf(float(x)) for x in row] for row in k]
        vv = [[mp.mpf(float(x)) for x in row] for row in v]
        for i in range(nq):
            qi = [mp.mpf(float(x)) for x in q[i]]
            n_i = nk if limits is None else int(limits[i])
            e = [mp.exp(sc * mp.fsum(a * b for a, b in zip(qi, kk[j]))) for j in range(n_i)]
            z = mp.fsum(e)
            for c in range(v.shape[1]):
                o[i, c] = float(mp.fsum(e[j] * vv[j][c] for j in range(n_i)) / z)
            lse[i] = float(mp.log(z))
    return o, lse
