"""The input prologue of a KDA layer, in numpy fp64: short convolution, Swish, L2 norm.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows Kimi K3 -- Architecture Notes, section 1.1: the q, k and v projections pass a
short convolution and then Swish, and q and k are then L2-normalised (the visualiser
page "Kimi K3" adds that the convolution has kernel size 4 and gives the local
context before the update). Per (token t, head h, channel c) of each projection x:

    conv_t = sum_{j=0..3} w[h, c, j] * x_{t-3+j}      (causal, depthwise, no bias)
    u_t    = Swish(conv_t) = conv_t * Sigmoid(conv_t)
    q_t    = u_t / sqrt(sum_c u_tc^2 + eps)            (q and k only; v keeps u_t)

Inputs before the start of a sequence are the sequence's convolution state (the
last three inputs of the text before it), or zeros. Readings where the pages are
silent: no bias; one weight row of 4 taps per (head, channel), tap 3 on the
current token; eps inside the square root; the state holds the three most recent
inputs in time order.

Layout: x [T_tot, H, d] per projection; weights [H, 2 d_k + d_v, 4] (the q
channels, then k, then v); convolution states [N, H, 3, 2 d_k + d_v] (time index
0 oldest).
"""

from __future__ import annotations

import numpy as np

# planted mistakes that the pins must catch
PROLOGUE_MUTATIONS = (
    "acausal",            # taps on t-2 .. t+1 instead of t-3 .. t
    "no_reset",           # the window runs across sequence boundaries
    "taps_reversed",      # tap 0 on the current token
    "norm_then_swish",    # Swish after the L2 norm
    "no_swish_v",         # v leaves the convolution without Swish
    "norm_v",             # v L2-normalised too
)


def _f64(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:
        pass
    return None if x is None else np.asarray(x, dtype=np.float64)


def swish(x):
    return x / (1.0 + np.exp(-x))


def l2_normalise(x, eps):
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def short_conv(x, w, cu_seqlens, state=None, mutation=None):
    """Causal depthwise convolution with 4 taps over each sequence of x [T, H, C].
    w [H, C, 4]; state [N, H, 3, C] or None. Returns (y [T, H, C], final state [N, H, 3, C])."""
    x = _f64(x)
    w = _f64(w)
    T, H, C = x.shape
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    N = cu.shape[0] - 1
    st = np.zeros((N, H, 3, C)) if state is None else _f64(state)
    y = np.zeros_like(x)
    final = np.zeros((N, H, 3, C))
    for n in range(N):
        bos, eos = int(cu[n]), int(cu[n + 1])
        prev = st[n]  # [H, 3, C], time order
        if mutation == "no_reset" and n > 0:
            prev = np.stack([x[bos - 3 + i] if bos - 3 + i >= 0 else np.zeros((H, C)) for i in range(3)], axis=1)
        # the sequence's inputs preceded by its state: index 3 + s is token bos + s
        ext = np.concatenate([prev.transpose(1, 0, 2), x[bos:eos]], axis=0)  # [3 + L, H, C]
        for s in range(eos - bos):
            acc = np.zeros((H, C))
            for j in range(4):
                if mutation == "acausal":
                    src = 3 + s - 2 + j
                    v = ext[src] if src < ext.shape[0] else np.zeros((H, C))
                else:
                    v = ext[3 + s - 3 + j]
                tap = 3 - j if mutation == "taps_reversed" else j
                acc += w[:, :, tap] * v
            y[bos + s] = acc
        final[n] = ext[-3:].transpose(1, 0, 2)
    return y, final


def kda_prologue(q_raw, k_raw, v_raw, conv_weight, cu_seqlens, conv_state=None, eps: float = 1e-6,
                 mutation: str | None = None):
    """ShortConv -> Swish (q, k, v) -> L2 norm (q, k). Returns (q, k, v, conv_final) in fp64."""
    if mutation is not None and mutation not in PROLOGUE_MUTATIONS:
        raise ValueError(f"unknown mutation {mutation!r}")
    q_raw, k_raw, v_raw = _f64(q_raw), _f64(k_raw), _f64(v_raw)
    dk, dv = q_raw.shape[-1], v_raw.shape[-1]
    w = _f64(conv_weight)
    if w.shape != (q_raw.shape[1], 2 * dk + dv, 4):
        raise ValueError("conv_weight must be [H, 2 d_k + d_v, 4]")
    x = np.concatenate([q_raw, k_raw, v_raw], axis=-1)
    conv, final = short_conv(x, w, cu_seqlens, conv_state, mutation)
    cq, ck, cv = conv[..., :dk], conv[..., dk:2 * dk], conv[..., 2 * dk:]
    if mutation == "norm_then_swish":
        q, k = swish(l2_normalise(cq, eps)), swish(l2_normalise(ck, eps))
    else:
        q, k = l2_normalise(swish(cq), eps), l2_normalise(swish(ck), eps)
    v = cv if mutation == "no_swish_v" else swish(cv)
    if mutation == "norm_v":
        v = l2_normalise(v, eps)
    return q, k, v, final
