"""Shared helpers for the parity tests: the tolerance metric and oracle calls."""

from __future__ import annotations

import os

import numpy as np
import torch

from oracle import kda_recurrent, kda_recurrent_gated

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
