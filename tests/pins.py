"""Pin checks for a KDA oracle, shared by the oracle tests and the planted-mistake tests.

Each check takes ``run(q, k, v, log_alpha, beta, cu_seqlens, lower_bound=, init_state=)``
returning ``(out, final_state)`` in fp64 numpy, and raises AssertionError when
the oracle disagrees with something the definition (Kimi K3 -- Architecture
Notes, section 1.1) or mathematics fixes independently of the oracle.
"""

from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

from oracle import kda_exact

NO_CLAMP = -1.0e300  # a lower bound no finite log-decay reaches


def rel_err(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    scale = max(float(np.sqrt(np.mean(b * b))), 1e-300)
    return float(np.max(np.abs(a - b))) / scale if a.size else 0.0


def _rng_rational(rng, lo, hi, den=16):
    return Fraction(int(rng.integers(int(lo * den), int(hi * den) + 1)), den)


def pin_exact_bruteforce(run, seed=0, cases=6):
    """Exact rational brute force with dense transition matrices, tiny sizes."""
    rng = np.random.default_rng(seed)
    for case in range(cases):
        dk = int(rng.integers(1, 4))
        dv = dk if case % 2 == 0 else int(rng.integers(1, 4))  # square cases catch axis mix-ups
        T = int(rng.integers(1, 7))
        q = [[_rng_rational(rng, -1, 1) for _ in range(dk)] for _ in range(T)]
        k = [[_rng_rational(rng, -1, 1) for _ in range(dk)] for _ in range(T)]
        v = [[_rng_rational(rng, -2, 2) for _ in range(dv)] for _ in range(T)]
        alpha = [[Fraction(int(rng.integers(1, 17)), 16) for _ in range(dk)] for _ in range(T)]
        beta = [Fraction(int(rng.integers(0, 17)), 16) for _ in range(T)]
        S0 = [[_rng_rational(rng, -1, 1) for _ in range(dv)] for _ in range(dk)]
        o_ex, S_ex = kda_exact(q, k, v, alpha, beta, S0)
        f = lambda m: np.array([[float(x) for x in row] for row in m], dtype=np.float64)
        la = np.log(f(alpha))[:, None, :]
        out, fin = run(f(q)[:, None, :], f(k)[:, None, :], f(v)[:, None, :], la,
                       np.array([float(b) for b in beta])[:, None], [0, T],
                       lower_bound=NO_CLAMP, init_state=f(S0)[None, None])
        assert rel_err(out[:, 0], f(o_ex)) < 1e-13, f"exact case {case}: outputs"
        assert rel_err(fin[0, 0], f(S_ex)) < 1e-13, f"exact case {case}: final state"


def _unit(rng, shape):
    x = rng.standard_normal(shape)
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def pin_identity_state(run, seed=1):
    """alpha = 1, beta = 0: the state never changes and o_t = S0^T q_t."""
    rng = np.random.default_rng(seed)
    T, dk, dv = 9, 5, 4
    q, k = _unit(rng, (T, 1, dk)), _unit(rng, (T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    S0 = rng.standard_normal((1, 1, dk, dv))
    out, fin = run(q, k, v, np.zeros((T, 1, dk)), np.zeros((T, 1)), [0, T], init_state=S0)
    assert rel_err(fin, S0) < 1e-15
    assert rel_err(out[:, 0], q[:, 0] @ S0[0, 0]) < 1e-14


def pin_pure_decay(run, seed=2):
    """beta = 0, any alpha: S_t = Diag(exp(sum g)) S0, o_t = S_t^T q_t."""
    rng = np.random.default_rng(seed)
    T, dk, dv = 7, 6, 3
    q, k = _unit(rng, (T, 1, dk)), _unit(rng, (T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    g = -rng.uniform(0.0, 2.0, (T, 1, dk))
    S0 = rng.standard_normal((1, 1, dk, dv))
    out, fin = run(q, k, v, g, np.zeros((T, 1)), [0, T], init_state=S0)
    G = np.cumsum(g[:, 0], axis=0)
    for t in range(T):
        St = np.exp(G[t])[:, None] * S0[0, 0]
        assert rel_err(out[t, 0], St.T @ q[t, 0]) < 1e-13
    assert rel_err(fin[0, 0], np.exp(G[-1])[:, None] * S0[0, 0]) < 1e-13


def pin_orthonormal_overwrite(run, seed=3):
    """alpha = 1, beta = 1, orthonormal keys: S_T^T k_j = v_j for every written key
    (exact overwrite) and the part of S0 orthogonal to span{k} is untouched."""
    rng = np.random.default_rng(seed)
    dk, dv, T = 8, 5, 6
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = Qm[:, :T].T  # T orthonormal rows
    q = _unit(rng, (T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    S0 = rng.standard_normal((1, 1, dk, dv))
    out, fin = run(q, keys[:, None, :], v, np.zeros((T, 1, dk)), np.ones((T, 1)), [0, T], init_state=S0)
    S = fin[0, 0]
    for j in range(T):
        assert rel_err(S.T @ keys[j], v[j, 0]) < 1e-12
    proj = np.eye(dk) - keys.T @ keys
    assert rel_err(proj @ S, proj @ S0[0, 0]) < 1e-12


def pin_scalar_recurrence(run, seed=4):
    """d_k = d_v = 1: s_t = (1 - b k^2) a s_{t-1} + b k v,  o_t = s_t q_t."""
    rng = np.random.default_rng(seed)
    T = 12
    q, k, v = rng.standard_normal(T), rng.standard_normal(T), rng.standard_normal(T)
    g = -rng.uniform(0.0, 3.0, T)
    b = rng.uniform(0.0, 1.0, T)
    s = 0.7
    o_ref = []
    for t in range(T):
        s = (1.0 - b[t] * k[t] ** 2) * math.exp(g[t]) * s + b[t] * k[t] * v[t]
        o_ref.append(s * q[t])
    out, fin = run(q[:, None, None], k[:, None, None], v[:, None, None], g[:, None, None], b[:, None],
                   [0, T], lower_bound=NO_CLAMP, init_state=np.full((1, 1, 1, 1), 0.7))
    assert rel_err(out[:, 0, 0], np.array(o_ref)) < 1e-13
    assert abs(fin[0, 0, 0, 0] - s) <= 1e-13 * max(1.0, abs(s))


def pin_lower_bound(run):
    """The retention factor never falls below exp(-5) ~ 6.7e-3 (Kimi K3 --
    Architecture Notes, section 1.2, the printed bound); values at or above
    the bound pass through unchanged."""
    dk, dv = 3, 2
    S0 = np.arange(1, dk * dv + 1, dtype=np.float64).reshape(1, 1, dk, dv)
    q = np.eye(dk)[:1][:, None, :]
    k = np.eye(dk)[1:2][:, None, :]
    v = np.zeros((1, 1, dv))
    la = np.array([[[-40.0, -5.0, -0.25]]])
    out, fin = run(q, k, v, la, np.zeros((1, 1)), [0, 1], lower_bound=-5.0, init_state=S0)
    ratio = fin[0, 0] / S0[0, 0]
    assert abs(ratio[0, 0] - 6.7e-3) < 0.05e-3 and abs(ratio[0, 0] - math.exp(-5.0)) < 1e-15
    assert abs(ratio[1, 0] - math.exp(-5.0)) < 1e-15
    assert abs(ratio[2, 0] - math.exp(-0.25)) < 1e-15


def pin_split_resume(run, seed=5):
    """prefill(x1 || x2) = prefill(x2; init = final(x1))."""
    rng = np.random.default_rng(seed)
    T, H, dk, dv, cut = 23, 2, 6, 4, 9
    q, k = _unit(rng, (T, H, dk)), _unit(rng, (T, H, dk))
    v = rng.standard_normal((T, H, dv))
    g = -np.logaddexp(0.0, rng.standard_normal((T, H, dk)))
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    S0 = 0.5 * rng.standard_normal((1, H, dk, dv))
    out, fin = run(q, k, v, g, b, [0, T], init_state=S0)
    o1, f1 = run(q[:cut], k[:cut], v[:cut], g[:cut], b[:cut], [0, cut], init_state=S0)
    o2, f2 = run(q[cut:], k[cut:], v[cut:], g[cut:], b[cut:], [0, T - cut], init_state=f1)
    assert rel_err(np.concatenate([o1, o2]), out) < 1e-13
    assert rel_err(f2, fin) < 1e-13


def pin_linearity(run, seed=6):
    """For fixed q, k, alpha, beta the map (V, S0) -> (O, S_T) is linear."""
    rng = np.random.default_rng(seed)
    T, dk, dv = 11, 5, 3
    q, k = _unit(rng, (T, 1, dk)), _unit(rng, (T, 1, dk))
    g = -rng.uniform(0.0, 1.0, (T, 1, dk))
    b = rng.uniform(0.0, 1.0, (T, 1))
    v1, v2 = rng.standard_normal((T, 1, dv)), rng.standard_normal((T, 1, dv))
    s1, s2 = rng.standard_normal((1, 1, dk, dv)), rng.standard_normal((1, 1, dk, dv))
    o1, f1 = run(q, k, v1, g, b, [0, T], init_state=s1)
    o2, f2 = run(q, k, v2, g, b, [0, T], init_state=s2)
    o3, f3 = run(q, k, 2.0 * v1 - 3.0 * v2, g, b, [0, T], init_state=2.0 * s1 - 3.0 * s2)
    assert rel_err(o3, 2.0 * o1 - 3.0 * o2) < 1e-12
    assert rel_err(f3, 2.0 * f1 - 3.0 * f2) < 1e-12


def pin_column_permutation(run, seed=7):
    """Each value column of S evolves on its own: permuting the columns of v and
    S0 permutes the columns of the outputs and of the final state."""
    rng = np.random.default_rng(seed)
    T, dk, dv = 10, 4, 6
    q, k = _unit(rng, (T, 1, dk)), _unit(rng, (T, 1, dk))
    g = -rng.uniform(0.0, 1.0, (T, 1, dk))
    b = rng.uniform(0.0, 1.0, (T, 1))
    v = rng.standard_normal((T, 1, dv))
    S0 = rng.standard_normal((1, 1, dk, dv))
    perm = rng.permutation(dv)
    o, f = run(q, k, v, g, b, [0, T], init_state=S0)
    op, fp = run(q, k, v[..., perm], g, b, [0, T], init_state=S0[..., perm])
    assert rel_err(op, o[..., perm]) < 1e-14
    assert rel_err(fp, f[..., perm]) < 1e-14


def pin_norm_bound(run, seed=8):
    """With |k| = 1, beta in [0,1], alpha <= 1: |S_t|_2 <= |S_{t-1}|_2 + beta_t |v_t|."""
    rng = np.random.default_rng(seed)
    T, dk, dv = 8, 5, 4
    q, k = _unit(rng, (T, 1, dk)), _unit(rng, (T, 1, dk))
    g = -rng.uniform(0.0, 0.5, (T, 1, dk))
    b = rng.uniform(0.0, 1.0, (T, 1))
    v = rng.standard_normal((T, 1, dv))
    S = rng.standard_normal((1, 1, dk, dv))
    for t in range(T):
        _, S_new = run(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1], b[t:t + 1], [0, 1], init_state=S)
        lhs = np.linalg.norm(S_new[0, 0], 2)
        rhs = np.linalg.norm(S[0, 0], 2) + b[t, 0] * np.linalg.norm(v[t, 0])
        assert lhs <= rhs * (1 + 1e-12)
        S = S_new


def pin_varlen_packing(run, seed=9):
    """Packing sequences with cu_seqlens equals running each one alone (including
    empty and length-1 sequences)."""
    rng = np.random.default_rng(seed)
    lengths = [5, 0, 1, 13, 2]
    H, dk, dv = 2, 4, 3
    T = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    q, k = _unit(rng, (T, H, dk)), _unit(rng, (T, H, dk))
    v = rng.standard_normal((T, H, dv))
    g = -np.logaddexp(0.0, rng.standard_normal((T, H, dk)))
    b = rng.uniform(0.0, 1.0, (T, H))
    S0 = rng.standard_normal((len(lengths), H, dk, dv))
    out, fin = run(q, k, v, g, b, cu, init_state=S0)
    for n, L in enumerate(lengths):
        a, e = cu[n], cu[n + 1]
        o_n, f_n = run(q[a:e], k[a:e], v[a:e], g[a:e], b[a:e], [0, L], init_state=S0[n:n + 1])
        assert rel_err(out[a:e], o_n) < 1e-15 if L else True
        assert rel_err(fin[n:n + 1], f_n) < 1e-15
    assert rel_err(fin[1], S0[1]) == 0.0  # an empty sequence hands its state through


ALL_PINS = [pin_exact_bruteforce, pin_identity_state, pin_pure_decay, pin_orthonormal_overwrite,
            pin_scalar_recurrence, pin_lower_bound, pin_split_resume, pin_linearity,
            pin_column_permutation, pin_norm_bound, pin_varlen_packing]
