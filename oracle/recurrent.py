"""ctypes front end of the fp64 C oracle (``kda_oracle.c``).

TEST INFRASTRUCTURE ONLY (see the package docstring). The C source is compiled
here with the host ``gcc`` on first use (or by ``__graft_entry__.build()``),
into ``oracle/_build/``. Definition followed: Kimi K3 -- Architecture Notes,
section 1.1, ``S_t = (I - b_t k_t k_t^T) Diag(a_t) S_{t-1} + b_t k_t v_t^T``,
``o_t = S_t^T q_t``, with ``log a_t`` clamped below at ``lower_bound``
(section 1.2), or, in the gated form of section 1.2 (the K3 row of its mapping
table), computed from decay logits ``z`` and per-head log-scales ``A_h`` as
``g = g_min * Sigmoid(e^{A_h} z)``, or, in the unbounded form of the earlier
models (the table's other row), as ``g = -e^{A_h} Softplus(z)``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libkda_oracle.so")

F64, F32, BF16 = 0, 1, 2

# planted mistakes understood by kda_oracle_recurrent_mutant (see kda_oracle.c)
MUTATIONS = {
    "no_decay": 1,
    "undecayed_prediction": 2,
    "sign": 3,
    "output_before_write": 4,
    "decay_value_axis": 5,
    "no_clamp": 6,
    "no_beta": 7,
}

# planted mistakes of the gated form, understood by kda_recurrent_gated(mutation=...)
GATE_MUTATIONS = {
    "gate_no_exp": 8,
    "gate_softplus": 9,
    "gate_sign": 10,
}

# planted mistakes of the unbounded form, understood by kda_recurrent_unbounded(mutation=...)
UNBOUNDED_MUTATIONS = {
    "unbounded_no_exp": 11,
    "unbounded_sign": 12,
    "unbounded_bounded_map": 13,
}

_lock = threading.Lock()
_lib = None


def oracle_library_path() -> str:
    return _LIB_PATH


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` into ``oracle/_build/libkda_oracle.so``."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            fn = lib.kda_oracle_recurrent_mutant
            vp, i32, i64, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
            fn.argtypes = [vp, vp, i32, vp, i32, vp, i32, vp, i32, vp, i64, i64, i64, i64,
                           f64, f64, vp, i32, vp, vp, i32, i32]
            fn.restype = i32
            fg = lib.kda_oracle_recurrent_gated
            fg.argtypes = [vp, vp, i32, vp, i32, vp, i32, vp, vp, i32, vp, i64, i64, i64, i64,
                           f64, f64, vp, i32, vp, vp, i32, i32]
            fg.restype = i32
            fu = lib.kda_oracle_recurrent_unbounded
            fu.argtypes = [vp, vp, i32, vp, i32, vp, i32, vp, vp, i32, vp, i64, i64, i64, i64,
                           f64, vp, i32, vp, vp, i32, i32]
            fu.restype = i32
            _lib = lib
    return _lib


def _as_array(x):
    """Return (contiguous numpy array, dtype code). bf16 torch tensors pass raw bits."""
    if x is None:
        return None, F64
    try:
        import torch  # only to accept torch CPU tensors without a copy through float
        if isinstance(x, torch.Tensor):
            x = x.detach()
            if x.device.type != "cpu":
                raise ValueError("oracle inputs must live on the CPU")
            if x.dtype == torch.bfloat16:
                return np.ascontiguousarray(x.contiguous().view(torch.int16).numpy()), BF16
            x = x.contiguous().numpy()
    except ImportError:
        pass
    x = np.asarray(x)
    if x.dtype == np.float64:
        return np.ascontiguousarray(x), F64
    if x.dtype == np.float32:
        return np.ascontiguousarray(x), F32
    if x.dtype in (np.int16, np.uint16):
        return np.ascontiguousarray(x), BF16
    return np.ascontiguousarray(x, dtype=np.float64), F64


def kda_recurrent_mutant(q, k, v, log_alpha, beta, cu_seqlens, *, mutation: int,
                         lower_bound: float = -5.0, scale: float = 1.0, init_state=None,
                         num_threads: int | None = None):
    """Run the oracle, optionally with one planted mistake (``mutation`` > 0).

    Shapes: q, k, log_alpha [T_tot, H, d_k]; v [T_tot, H, d_v]; beta [T_tot, H];
    cu_seqlens [N+1] (int); init_state [N, H, d_k, d_v] or None (zeros).
    Returns (out [T_tot, H, d_v], final_state [N, H, d_k, d_v]) as float64.
    """
    lib = _load()
    qa, dt_qk = _as_array(q)
    ka, dt_k = _as_array(k)
    if dt_k != dt_qk:
        raise ValueError("q and k must share one element type")
    va, dt_v = _as_array(v)
    la, dt_la = _as_array(log_alpha)
    ba, dt_b = _as_array(beta)
    ia, dt_i = _as_array(init_state)
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    T_tot, H, dk = qa.shape
    dv = va.shape[-1]
    N = cu.shape[0] - 1
    if ka.shape != (T_tot, H, dk) or la.shape != (T_tot, H, dk) or va.shape[:2] != (T_tot, H):
        raise ValueError("q/k/log_alpha/v shapes disagree")
    if ba.shape != (T_tot, H):
        raise ValueError("beta must be [T_tot, H]")
    if ia is not None and ia.shape != (N, H, dk, dv):
        raise ValueError("init_state must be [N, H, d_k, d_v]")
    if N < 0 or cu[0] != 0 or cu[-1] != T_tot:
        raise ValueError("cu_seqlens must start at 0 and end at T_tot")
    out = np.zeros((T_tot, H, dv), dtype=np.float64)
    final = np.zeros((N, H, dk, dv), dtype=np.float64)
    nt = num_threads or os.cpu_count() or 1

    def ptr(a):
        return None if a is None else a.ctypes.data

    rc = lib.kda_oracle_recurrent_mutant(
        ptr(qa), ptr(ka), dt_qk, ptr(va), dt_v, ptr(la), dt_la, ptr(ba), dt_b, ptr(cu), N, H, dk, dv,
        float(lower_bound), float(scale), ptr(ia), dt_i, ptr(out), ptr(final), int(nt), int(mutation))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_recurrent failed with code {rc}")
    return out, final


def kda_recurrent(q, k, v, log_alpha, beta, cu_seqlens, *, lower_bound: float = -5.0,
                  scale: float = 1.0, init_state=None, num_threads: int | None = None):
    """fp64 token-by-token KDA recurrence; see ``kda_recurrent_mutant``."""
    return kda_recurrent_mutant(q, k, v, log_alpha, beta, cu_seqlens, mutation=0,
                                lower_bound=lower_bound, scale=scale, init_state=init_state,
                                num_threads=num_threads)


def kda_recurrent_unbounded(q, k, v, z, A_log, beta, cu_seqlens, *, scale: float = 1.0, init_state=None,
                            num_threads: int | None = None, mutation: int = 0):
    """fp64 KDA recurrence with the unbounded log-decay ``g = -e^{A_h} Softplus(z)`` of the earlier
    models (Kimi K3 -- Architecture Notes, section 1.2, the GDN / Mamba-2 / Kimi Linear row of the
    mapping table). Arguments as in ``kda_recurrent_gated`` (no g_min); ``mutation`` may be one of
    ``UNBOUNDED_MUTATIONS``."""
    return _run_gate(q, k, v, z, A_log, beta, cu_seqlens, None, scale, init_state, num_threads, mutation)


def kda_recurrent_gated(q, k, v, z, A_log, beta, cu_seqlens, *, g_min: float = -5.0, scale: float = 1.0,
                        init_state=None, num_threads: int | None = None, mutation: int = 0):
    """fp64 KDA recurrence with the gated log-decay ``g = g_min * Sigmoid(e^{A_h} z)``.

    z [T_tot, H, d_k] (float or bf16 bits, like q/k); A_log [H]; other arguments as in
    ``kda_recurrent_mutant``. ``mutation`` may be one of ``GATE_MUTATIONS`` (or 1, no decay).
    Returns (out [T_tot, H, d_v], final_state [N, H, d_k, d_v]) as float64.
    """
    return _run_gate(q, k, v, z, A_log, beta, cu_seqlens, g_min, scale, init_state, num_threads, mutation)


def _run_gate(q, k, v, z, A_log, beta, cu_seqlens, g_min, scale, init_state, num_threads, mutation):
    """Both gated forms: the bounded map with ``g_min``, the unbounded one when it is None."""
    lib = _load()
    qa, dt_qk = _as_array(q)
    ka, dt_k = _as_array(k)
    if dt_k != dt_qk:
        raise ValueError("q and k must share one element type")
    va, dt_v = _as_array(v)
    za, dt_z = _as_array(z)
    ba, dt_b = _as_array(beta)
    ia, dt_i = _as_array(init_state)
    try:
        import torch
        if isinstance(A_log, torch.Tensor):
            A_log = A_log.detach().cpu().double().numpy()
    except ImportError:
        pass
    aa = np.ascontiguousarray(np.asarray(A_log, dtype=np.float64))
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    T_tot, H, dk = qa.shape
    dv = va.shape[-1]
    N = cu.shape[0] - 1
    if ka.shape != (T_tot, H, dk) or za.shape != (T_tot, H, dk) or va.shape[:2] != (T_tot, H):
        raise ValueError("q/k/z/v shapes disagree")
    if aa.shape != (H,):
        raise ValueError("A_log must be [H]")
    if ba.shape != (T_tot, H):
        raise ValueError("beta must be [T_tot, H]")
    if ia is not None and ia.shape != (N, H, dk, dv):
        raise ValueError("init_state must be [N, H, d_k, d_v]")
    if N < 0 or cu[0] != 0 or cu[-1] != T_tot:
        raise ValueError("cu_seqlens must start at 0 and end at T_tot")
    out = np.zeros((T_tot, H, dv), dtype=np.float64)
    final = np.zeros((N, H, dk, dv), dtype=np.float64)
    nt = num_threads or os.cpu_count() or 1

    def ptr(a):
        return None if a is None else a.ctypes.data

    if g_min is None:
        rc = lib.kda_oracle_recurrent_unbounded(
            ptr(qa), ptr(ka), dt_qk, ptr(va), dt_v, ptr(za), dt_z, ptr(aa), ptr(ba), dt_b, ptr(cu), N, H, dk, dv,
            float(scale), ptr(ia), dt_i, ptr(out), ptr(final), int(nt), int(mutation))
    else:
        rc = lib.kda_oracle_recurrent_gated(
            ptr(qa), ptr(ka), dt_qk, ptr(va), dt_v, ptr(za), dt_z, ptr(aa), ptr(ba), dt_b, ptr(cu), N, H, dk, dv,
            float(g_min), float(scale), ptr(ia), dt_i, ptr(out), ptr(final), int(nt), int(mutation))
    if rc != 0:
        raise RuntimeError(f"the gated oracle failed with code {rc}")
    return out, final
