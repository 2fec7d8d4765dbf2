"""Exact rational brute force of the KDA recurrence for tiny inputs.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows Kimi K3 -- Architecture Notes, section 1.1 literally: each step builds
the dense transition matrix M_t = (I - beta_t k_t k_t^T) Diag(alpha_t) and the
write matrix beta_t k_t v_t^T, then S_t = M_t S_{t-1} + beta_t k_t v_t^T and
o_t = S_t^T q_t. Retention factors alpha are given directly (no exp), so every
number stays a ``fractions.Fraction`` and the result is exact.
"""

from __future__ import annotations

from fractions import Fraction


def _matmul(X, Y):
    return [[sum((X[i][m] * Y[m][j] for m in range(len(Y))), Fraction(0)) for j in range(len(Y[0]))]
            for i in range(len(X))]


def kda_exact(q, k, v, alpha, beta, S0=None):
    """One head, one sequence. q, k, alpha: T lists of d_k numbers; v: T lists of
    d_v numbers; beta: T numbers; S0: d_k x d_v (zeros if None). Returns (o, S_T)
    as nested lists of Fractions: o is T x d_v, S_T is d_k x d_v."""
    T = len(q)
    dk = len(k[0]) if T else len(S0)
    dv = len(v[0]) if T else len(S0[0])
    F = Fraction
    S = [[F(0)] * dv for _ in range(dk)] if S0 is None else [[F(x) for x in row] for row in S0]
    outs = []
    for t in range(T):
        kt = [F(x) for x in k[t]]
        qt = [F(x) for x in q[t]]
        vt = [F(x) for x in v[t]]
        at = [F(x) for x in alpha[t]]
        bt = F(beta[t])
        # M_t = (I - b k k^T) Diag(a): entry (i, j) = (delta_ij - b k_i k_j) a_j
        M = [[((F(1) if i == j else F(0)) - bt * kt[i] * kt[j]) * at[j] for j in range(dk)]
             for i in range(dk)]
        MS = _matmul(M, S)
        S = [[MS[i][j] + bt * kt[i] * vt[j] for j in range(dv)] for i in range(dk)]
        outs.append([sum((S[i][j] * qt[i] for i in range(dk)), F(0)) for j in range(dv)])
    return outs, S
