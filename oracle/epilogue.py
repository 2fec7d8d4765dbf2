"""Output gate with head-wise RMSNorm, in numpy fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows Kimi K3 -- Architecture Notes, section 1.3 "Full-rank output gate": the
recurrent read-out o_t of each head is RMS-normalised, then multiplied by the
sigmoid of a full-rank, input-dependent gate, before the output projection:
y = W_o [Sigmoid(W_g x) (.) RMSNorm(o)]. The two projections W_g and W_o are
matmuls outside the recurrence; this function takes the gate logits r = W_g x
as an input and returns the bracket, per token and head:

    out[t, h, :] = Sigmoid(r[t, h, :]) * w * o[t, h, :] / sqrt(mean_j o[t, h, j]^2 + eps)

Readings where the page is silent: the RMSNorm runs over the d_v channels of one
(token, head) pair ("head-wise"), with a learnable per-channel weight w [d_v]
shared by the heads (ones when absent) and a small eps inside the square root,
as in the usual definition of RMSNorm; o includes the read-out's ``scale``.
"""

from __future__ import annotations

import numpy as np

# planted mistakes that the pins must catch
EPILOGUE_MUTATIONS = (
    "sum_not_mean",       # divide by sqrt(sum of squares) instead of the mean
    "norm_over_heads",    # one RMS over all heads of a token
    "norm_over_tokens",   # one RMS over all tokens of a head, per channel
    "no_sigmoid",         # the raw logits multiply the output
    "sigmoid_sign",       # Sigmoid(-r)
    "eps_outside",        # sqrt(mean) + eps
    "no_weight",          # w ignored
)


def _f64(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:
        pass
    return np.asarray(x, dtype=np.float64)


def output_gate_rmsnorm(o, r, weight=None, eps: float = 1e-6, mutation: str | None = None):
    """o, r [..., H, d_v] (read-out and gate logits); weight [d_v] or None; returns float64."""
    o = _f64(o)
    r = _f64(r)
    if o.shape != r.shape:
        raise ValueError("o and the gate logits must have one shape")
    if mutation is not None and mutation not in EPILOGUE_MUTATIONS:
        raise ValueError(f"unknown mutation {mutation!r}")
    dv = o.shape[-1]
    w = np.ones(dv) if weight is None else _f64(weight)
    if w.shape != (dv,):
        raise ValueError("weight must be [d_v]")
    if mutation == "no_weight":
        w = np.ones(dv)

    sq = o * o
    if mutation == "sum_not_mean":
        ms = sq.sum(axis=-1, keepdims=True)
    elif mutation == "norm_over_heads":
        ms = sq.mean(axis=(-2, -1), keepdims=True)
    elif mutation == "norm_over_tokens":
        ms = sq.mean(axis=0, keepdims=True)
    else:
        ms = sq.mean(axis=-1, keepdims=True)
    if mutation == "eps_outside":
        normed = o / (np.sqrt(ms) + eps)
    else:
        normed = o / np.sqrt(ms + eps)

    if mutation == "no_sigmoid":
        gate = r
    elif mutation == "sigmoid_sign":
        gate = 1.0 / (1.0 + np.exp(r))
    else:
        gate = 1.0 / (1.0 + np.exp(-r))
    return gate * w * normed
