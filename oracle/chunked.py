"""Chunkwise form of the KDA recurrence, numpy fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Kimi K3 -- Architecture Notes, section 1.2 ("The problem") says the kernel is
recurrent across chunks and parallel within each chunk, with keys rescaled by
cumulative decay. The pages print no chunked equations; they are derived here
from the section 1.1 recurrence and kept free of any blocking or tiling trick:

Within one chunk entered with state S0, let G_t be the running sum of the
clamped log-decays g (t counted from the chunk start) and Gamma_t = exp(G_t).
Unrolling the recurrence gives

    S_r = Diag(Gamma_r) S0 + sum_{i<=r} Diag(Gamma_r / Gamma_i) k_i u_i^T,
    u_t + sum_{i<t} A[t,i] u_i = beta_t (v_t - S0^T (Gamma_t * k_t)),
    A[t,i] = beta_t sum_c k_tc k_ic exp(G_tc - G_ic)            (i < t),

so with T = (I + A)^{-1} (unit lower triangular; the "UT/WY" transform)

    U   = T Diag(beta) V - T Diag(beta) (K * Gamma) S0  =  U~ - W S0,
    O   = (Q * Gamma) S0 + P U,   P[t,i] = sum_c q_tc k_ic exp(G_tc - G_ic)  (i <= t),
    S_C = Diag(Gamma_last) S0 + (K * exp(G_last - G))^T U.

The inverse is a library call (numpy.linalg.inv); exp(G_t - G_i) is formed
directly from the difference, so no scaling factor can overflow in fp64.
"""

from __future__ import annotations

import numpy as np


def _f64(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", dtype=torch.float64).numpy()
    except ImportError:
        pass
    return np.asarray(x, dtype=np.float64)


def chunk_quantities(q, k, v, g, beta):
    """All intra-chunk quantities of one chunk of one head, in fp64.

    q, k, g: [L, d_k]; v: [L, d_v]; beta: [L]; g is the already clamped log-decay.
    Returns a dict with G, Gamma, A, T, P, W, U_tilde, Kd (= K * exp(G_last - G)).
    """
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    L = q.shape[0]
    G = np.cumsum(g, axis=0)
    Gamma = np.exp(G)
    tri_strict = np.tril(np.ones((L, L), dtype=bool), -1)
    tri_incl = np.tril(np.ones((L, L), dtype=bool), 0)
    # relative decay exp(G_t - G_i) for every (t, i, channel), kept only where i <= t
    diff = G[:, None, :] - G[None, :, :]
    decay = np.where(tri_incl[:, :, None], np.exp(np.where(tri_incl[:, :, None], diff, 0.0)), 0.0)
    A = beta[:, None] * np.einsum("tc,ic,tic->ti", k, k, decay)
    A = np.where(tri_strict, A, 0.0)
    P = np.where(tri_incl, np.einsum("tc,ic,tic->ti", q, k, decay), 0.0)
    T = np.linalg.inv(np.eye(L) + A)
    W = T @ (beta[:, None] * k * Gamma)
    U_tilde = T @ (beta[:, None] * v)
    Kd = k * np.exp(G[-1][None, :] - G)
    return {"G": G, "Gamma": Gamma, "A": A, "T": T, "P": P, "W": W, "U_tilde": U_tilde, "Kd": Kd}


def kda_chunked(q, k, v, log_alpha, beta, cu_seqlens, *, chunk: int = 64, lower_bound: float = -5.0,
                scale: float = 1.0, init_state=None):
    """KDA prefill in chunkwise form; same shapes and results as ``kda_recurrent``.

    Chunks restart at every sequence start; the last chunk of a sequence may be
    shorter than ``chunk``.
    """
    q, k, v, log_alpha, beta = (_f64(x) for x in (q, k, v, log_alpha, beta))
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    T_tot, H, dk = q.shape
    dv = v.shape[-1]
    N = cu.shape[0] - 1
    init = None if init_state is None else _f64(init_state)
    g_all = np.where(log_alpha < lower_bound, lower_bound, log_alpha)
    out = np.zeros((T_tot, H, dv))
    final = np.zeros((N, H, dk, dv))
    for n in range(N):
        for h in range(H):
            S = np.zeros((dk, dv)) if init is None else init[n, h].copy()
            for s0 in range(int(cu[n]), int(cu[n + 1]), chunk):
                s1 = min(s0 + chunk, int(cu[n + 1]))
                cq = chunk_quantities(q[s0:s1, h], k[s0:s1, h], v[s0:s1, h], g_all[s0:s1, h], beta[s0:s1, h])
                U = cq["U_tilde"] - cq["W"] @ S
                O = (q[s0:s1, h] * cq["Gamma"]) @ S + cq["P"] @ U
                out[s0:s1, h] = scale * O
                S = cq["Gamma"][-1][:, None] * S + cq["Kd"].T @ U
            final[n, h] = S
    return out, final
