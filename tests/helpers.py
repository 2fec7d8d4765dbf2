"""Shared helpers for the parity tests: the tolerance metric and oracle calls."""

from __future__ import annotations

import os

import numpy as np
import torch

from oracle import kda_recurrent, kda_recurrent_gated, output_gate_rmsnorm

# Tolerances on max|gpu - oracle| / rms(oracle), per tensor: fp32 inputs, and
# bf16 inputs with fp32 state.
TOL_F32 = 1e-4
TOL_BF16 = 2e-2


def rel_max_err(gpu, ref) -> float:
    g = np.asarray(gpu.detach().to("cpu", torch.float64).numpy() if isinstance(gpu, torch.Tensor) else gpu,
                   dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    if r.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(r * r)))
    return float(np.max(np.abs(g - r))) / max(rms, 1e-30)


def cpu(t):
    return None if t is None else t.detach().to("cpu")


def oracle_prefill(case, lower_bound=-5.0, scale=1.0, threads=None):
    """fp64 oracle on exactly the tensors of a PrefillCase (moved to the CPU)."""
    return kda_recurrent(cpu(case.q), cpu(case.k), cpu(case.v), cpu(case.log_alpha), cpu(case.beta),
                         cpu(case.cu_seqlens).to(torch.int64).numpy(), lower_bound=lower_bound, scale=scale,
                         init_state=cpu(case.init_state), num_threads=threads or os.cpu_count())


def oracle_prefill_gated(case, g_min=-5.0, scale=1.0, threads=None, heads=None):
    """fp64 oracle of the gated form on a gated PrefillCase (optionally on a subset of heads)."""
    sel = (lambda t: t) if heads is None else (lambda t: t[:, heads].contiguous())
    A = case.A_log if heads is None else case.A_log[heads]
    init = case.init_state if (heads is None or case.init_state is None) else case.init_state[:, heads].contiguous()
    return kda_recurrent_gated(cpu(sel(case.q)), cpu(sel(case.k)), cpu(sel(case.v)), cpu(sel(case.z)), cpu(A),
                               cpu(sel(case.beta)), cpu(case.cu_seqlens).to(torch.int64).numpy(), g_min=g_min,
                               scale=scale, init_state=cpu(init), num_threads=threads or os.cpu_count())


def tol_for(dtype) -> float:
    return TOL_BF16 if dtype == torch.bfloat16 else TOL_F32


def oracle_prefill_out_gate(case, bound=-5.0, scale=1.0, eps=1e-6, threads=None, weight=True):
    """fp64 oracle of a prefill with the output gate: the recurrence (clamped, or gated when the
    case carries z), then Sigmoid(r) * w * o / sqrt(mean(o^2) + eps) per token and head.
    Returns (y, final_state, o): o is the read-out before the gate."""
    if case.z is not None:
        o, f = oracle_prefill_gated(case, g_min=bound, scale=scale, threads=threads)
    else:
        o, f = oracle_prefill(case, lower_bound=bound, scale=scale, threads=threads)
    w = cpu(case.norm_weight) if weight else None
    return output_gate_rmsnorm(o, cpu(case.out_gate), w, eps), f, o


def gated_output_err(y, y_ref, o_ref, bf16_out=False) -> float:
    """Error of an output-gated result: max |y - y_ref| / rms(y_ref), where each (token, head)
    row's error is first multiplied by min(1, rms_row(o_ref) / rms(o_ref)).

    The RMSNorm divides a row of the read-out by its own RMS, so an absolute read-out error
    e reaches y as e / rms_row(o): on a row whose read-out is 100 times smaller than typical,
    the same kernel error shows up 100 times larger. Scaling such rows back by
    rms_row / rms bounds y by exactly the read-out's own metric max |do| / rms(o). A bf16
    output adds one rounding, 2^-8 |y_ref|, per element."""
    g = np.asarray(y.detach().to("cpu", torch.float64).numpy() if isinstance(y, torch.Tensor) else y)
    d = np.abs(g - y_ref)
    if bf16_out:
        d = np.maximum(d - 2.0 ** -8 * np.abs(y_ref), 0.0)
    rms_o = float(np.sqrt(np.mean(o_ref * o_ref)))
    row = np.sqrt(np.mean(o_ref * o_ref, axis=-1, keepdims=True))
    d = d * np.minimum(1.0, row / max(rms_o, 1e-300))
    return float(d.max()) / max(float(np.sqrt(np.mean(y_ref * y_ref))), 1e-300) if d.size else 0.0
