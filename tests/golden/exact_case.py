"""Exact rational mLSTM example (no oracle, no CUDA): the unrolled sum of section 3
"The Parallel Dual Form" of the llms.blog xLSTM page, evaluated with fractions."""
from fractions import Fraction

import numpy as np


def exact_rational_case():
    """Integer q, k, v with f~ = 0 (f = 1/2) and i~ = 0 (i = 1), d_qk = 4 (scale 1/2):
    C_t = sum_j 2^{-(t-j)} v_j (k_j/2)^T exactly; returns the inputs and exact h, C, n."""
    rng = np.random.default_rng(2)
    S, DQK, DV = 6, 4, 3
    q = rng.integers(-3, 4, (1, 1, S, DQK)).astype(np.float64)
    k = rng.integers(-3, 4, (1, 1, S, DQK)).astype(np.float64)
    v = rng.integers(-3, 4, (1, 1, S, DV)).astype(np.float64)
    ig = np.zeros((1, 1, S))
    fg = np.zeros((1, 1, S))
    Fr = Fraction
    h = [[Fr(0)] * DV for _ in range(S)]
    C = [[Fr(0)] * DQK for _ in range(DV)]
    n = [Fr(0)] * DQK
    for t in range(S):
        C = [[Fr(0)] * DQK for _ in range(DV)]
        n = [Fr(0)] * DQK
        for j in range(t + 1):
            wgt = Fr(1, 2 ** (t - j))  # (prod_{tau=j+1..t} 1/2) * i_j
            for a in range(DV):
                for c in range(DQK):
                    C[a][c] += wgt * Fr(int(v[0, 0, j, a])) * Fr(int(k[0, 0, j, c]), 2)
            for c in range(DQK):
                n[c] += wgt * Fr(int(k[0, 0, j, c]), 2)
        nq = sum(n[c] * Fr(int(q[0, 0, t, c])) for c in range(DQK))
        den = max(abs(nq), Fr(1))
        for a in range(DV):
            h[t][a] = sum(C[a][c] * Fr(int(q[0, 0, t, c])) for c in range(DQK)) / den
    return (q, k, v, ig, fg), h, C, n
