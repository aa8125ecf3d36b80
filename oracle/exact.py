"""Exact rational evaluation of the gated delta rule for tiny cases.

TEST INFRASTRUCTURE ONLY.  The token recurrence of the FlashQLA blog ("Further
optimisation via gate decay") with a multiplicative decay alpha_t supplied
directly as a rational (so no logarithm is involved), written out with Python
``fractions.Fraction`` matrices:

    S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
    o_t = scale * S_t^T q_t

Used to brute-force T <= 8, dk, dv <= 4 cases and to write the golden
fixtures under ``tests/golden/``.
"""
from __future__ import annotations

from fractions import Fraction


def _mat(rows, cols, fill=Fraction(0)):
    return [[fill for _ in range(cols)] for _ in range(rows)]


def exact_recurrence(q, k, v, alpha, beta, scale, S0=None):
    """q, k: T lists of dk Fractions; v: T lists of dv Fractions; alpha, beta:
    T Fractions (alpha may instead be T lists of dk Fractions for a
    per-key-channel decay); scale: Fraction; S0: dk x dv list or None.
    Returns (o: T lists of dv Fractions, S_T: dk x dv list)."""
    T = len(q)
    dk, dv = len(k[0]), len(v[0])
    S = _mat(dk, dv) if S0 is None else [[Fraction(x) for x in row] for row in S0]
    outs = []
    for t in range(T):
        a = alpha[t]
        a_vec = list(a) if isinstance(a, (list, tuple)) else [a] * dk
        # P = Diag(alpha) (I - beta k k^T): P[i][j] = a_i (delta_ij - beta k_i k_j)
        P = [[a_vec[i] * ((1 if i == j else 0) - beta[t] * k[t][i] * k[t][j])
              for j in range(dk)] for i in range(dk)]
        # For a scalar decay Diag(alpha) commutes with (I - beta k k^T); for the
        # per-channel decay the recurrence is (I - beta k k^T) Diag(alpha) S.
        if isinstance(a, (list, tuple)):
            D = [[a_vec[i] * S[i][j] for j in range(dv)] for i in range(dk)]
            newS = [[sum(((1 if i == m else 0) - beta[t] * k[t][i] * k[t][m]) * D[m][j]
                         for m in range(dk)) for j in range(dv)] for i in range(dk)]
        else:
            newS = [[sum(P[i][m] * S[m][j] for m in range(dk)) for j in range(dv)]
                    for i in range(dk)]
        for i in range(dk):
            for j in range(dv):
                newS[i][j] += beta[t] * k[t][i] * v[t][j]
        S = newS
        outs.append([scale * sum(S[i][j] * q[t][i] for i in range(dk)) for j in range(dv)])
    return outs, S
