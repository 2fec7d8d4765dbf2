"""Thin Python binding of libkda (include/kda.h) over ctypes.

Argument marshalling only: every step of prefill and decode runs in the CUDA
kernels of ``libkda.so``. Tensors are torch CUDA tensors (PyTorch provides the
device memory and the stream); the functions check shapes and dtypes, pass raw
pointers, and raise ``KdaError`` on any non-OK status. There is no CPU
fallback: if ``libkda.so`` has not been built, importing the library raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkda.so")
ROOT = os.path.dirname(_HERE)
HEADERS = [os.path.join(ROOT, "include", "kda.h"), os.path.join(ROOT, "include", "kda_selftest.h")]

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_TIMEOUT, KDA_ERR_RANGE = 0, 1, 2, 3, 4, 5
KDA_F32, KDA_BF16 = 0, 1

_lock = threading.Lock()
_lib = None


KDA_DECAY_CLAMPED, KDA_DECAY_GATED, KDA_DECAY_UNBOUNDED = 0, 1, 2


class PrefillParams(ctypes.Structure):
    """``kda_prefill_params`` of include/kda.h, field for field."""
    _fields_ = [("struct_size", ctypes.c_uint32), ("in_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
                ("decay_form", ctypes.c_int32), ("num_seqs", ctypes.c_int32), ("H", ctypes.c_int32),
                ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32), ("total_tokens", ctypes.c_int64),
                ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("decay", ctypes.c_void_p),
                ("A_log", ctypes.c_void_p), ("beta", ctypes.c_void_p), ("cu_seqlens", ctypes.c_void_p),
                ("init_state", ctypes.c_void_p), ("out_gate", ctypes.c_void_p), ("norm_weight", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("final_state", ctypes.c_void_p), ("decay_bound", ctypes.c_float),
                ("scale", ctypes.c_float), ("norm_eps", ctypes.c_float), ("force_recurrent", ctypes.c_int32),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)]


class DecodeParams(ctypes.Structure):
    """``kda_decode_params`` of include/kda.h, field for field."""
    _fields_ = [("struct_size", ctypes.c_uint32), ("in_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
                ("decay_form", ctypes.c_int32), ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("d_k", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("decay", ctypes.c_void_p), ("A_log", ctypes.c_void_p), ("beta", ctypes.c_void_p),
                ("state", ctypes.c_void_p), ("out_gate", ctypes.c_void_p), ("norm_weight", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("conv_weight", ctypes.c_void_p), ("conv_state", ctypes.c_void_p),
                ("decay_bound", ctypes.c_float), ("scale", ctypes.c_float), ("norm_eps", ctypes.c_float),
                ("l2_eps", ctypes.c_float)]


class KdaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what} failed: {status_string(status)}")


def _declare(lib):
    vp, i32, i64, f32, u32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_uint32
    sz = ctypes.c_size_t
    prefill_args = [vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, i32, i32, f32, f32, vp, vp, vp, vp]
    lib.kda_prefill.argtypes = prefill_args[:-1] + [vp, sz, vp]
    lib.kda_prefill.restype = i32
    lib.kda_prefill_workspace_size.argtypes = [i64, i32, i32, i32, i32]
    lib.kda_prefill_workspace_size.restype = sz
    lib.kda_prefill_recurrent.argtypes = prefill_args
    lib.kda_prefill_noalloc.argtypes = prefill_args
    lib.kda_prefill_noalloc.restype = i32
    lib.kda_prefill_recurrent.restype = i32
    lib.kda_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, f32, vp]
    lib.kda_decode.restype = i32
    gated_args = [vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, i32, i32, f32, f32, vp, vp, vp, vp]
    lib.kda_prefill_gated.argtypes = gated_args
    lib.kda_prefill_gated.restype = i32
    lib.kda_prefill_gated_recurrent.argtypes = gated_args
    lib.kda_prefill_gated_recurrent.restype = i32
    lib.kda_decode_gated.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, f32, vp]
    lib.kda_decode_gated.restype = i32
    lib.kda_prefill_ex.argtypes = [ctypes.POINTER(PrefillParams), vp]
    lib.kda_prefill_ex.restype = i32
    lib.kda_decode_ex.argtypes = [ctypes.POINTER(DecodeParams), vp]
    lib.kda_decode_ex.restype = i32
    lib.kda_prologue.argtypes = [vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, i32, vp, f32, vp, vp, vp, vp, vp]
    lib.kda_prologue.restype = i32
    lib.kda_check_device_error.argtypes = [vp]
    lib.kda_check_device_error.restype = i32
    lib.kda_status_string.argtypes = [i32]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_version.argtypes = []
    lib.kda_version.restype = i32
    lib.kda_selftest_umma.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, u32, u32, u32, u32, vp, vp]
    lib.kda_selftest_umma.restype = i32
    lib.kda_selftest_wait_timeout.argtypes = [vp, vp]
    lib.kda_selftest_wait_timeout.restype = i32


def lib():
    """The loaded libkda (loaded once). Raises if the library was not built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                                   "(the KDA kernels have no fallback)")
            handle = ctypes.CDLL(LIB_PATH)
            _declare(handle)
            _lib = handle
    return _lib


def status_string(status: int) -> str:
    return lib().kda_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _io_dtype(dtype) -> int:
    if dtype == torch.bfloat16:
        return KDA_BF16
    if dtype == torch.float32:
        return KDA_F32
    raise TypeError(f"q/k/v and out must be bfloat16 or float32, got {dtype}")


def _check_cuda(*tensors):
    for t in tensors:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("KDA tensors must be contiguous CUDA tensors")


def workspace_size(total_tokens: int, num_seqs: int, H: int, d_k: int = 128, d_v: int = 128) -> int:
    """Bytes of device scratch ``kda_prefill`` can use for these sizes (``kda_prefill_workspace_size``)."""
    return int(lib().kda_prefill_workspace_size(int(total_tokens), int(num_seqs), int(H), int(d_k), int(d_v)))


def _workspace(workspace, T, N, H, d_k, d_v, device):
    """(pointer, bytes) of the scratch handed to the library: ``"auto"`` allocates what
    ``kda_prefill_workspace_size`` asks for (through torch's caching allocator), ``None`` passes
    none (one CTA per chain), a uint8 CUDA tensor is passed as given."""
    if workspace is None:
        return None, 0
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError("workspace must be 'auto', None or a uint8 CUDA tensor")
        n = workspace_size(T, N, H, d_k, d_v)
        if n == 0:
            return None, 0
        workspace = torch.empty(n, dtype=torch.uint8, device=device)
    _check_cuda(workspace)
    return ctypes.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size()


def prefill(q, k, v, log_alpha, beta, cu_seqlens, init_state=None, *, out=None, final_state=None,
            out_dtype=torch.float32, lower_bound: float = -5.0, scale: float = 1.0, stream=None,
            recurrent: bool = False, want_final: bool = True, workspace="auto"):
    """KDA prefill over packed variable-length sequences (``kda_prefill``).

    q, k [T, H, d_k], v [T, H, d_v] (bf16 or fp32, one dtype); log_alpha [T, H, d_k] fp32;
    beta [T, H] fp32; cu_seqlens [N+1] int32 (device); init_state [N, H, d_k, d_v] fp32 or None.
    Returns (out [T, H, d_v] in ``out_dtype`` (or out's dtype), final_state [N, H, d_k, d_v] or
    None). ``recurrent=True`` forces the fp32 token-recurrent kernel (``kda_prefill_recurrent``).
    ``workspace``: see ``_workspace`` (the default lets the library pick its parallel schedule).
    """
    T, H, d_k = q.shape
    d_v = v.shape[-1]
    N = cu_seqlens.shape[0] - 1
    dt = _io_dtype(q.dtype)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    if log_alpha.dtype != torch.float32 or beta.dtype != torch.float32:
        raise TypeError("log_alpha and beta must be float32")
    if cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    if out is None:
        out = torch.empty((T, H, d_v), dtype=out_dtype, device=q.device)
    odt = _io_dtype(out.dtype)
    if final_state is None and want_final:
        final_state = torch.empty((N, H, d_k, d_v), dtype=torch.float32, device=q.device)
    _check_cuda(q, k, v, log_alpha, beta, cu_seqlens, init_state, out, final_state)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(cu_seqlens), N, T, H, d_k, d_v, dt,
            odt, float(lower_bound), float(scale), _ptr(init_state), _ptr(out), _ptr(final_state))
    if recurrent:
        st = lib().kda_prefill_recurrent(*args, _stream_handle(stream))
    else:
        ws, ws_bytes = _workspace(workspace, T, N, H, d_k, d_v, q.device)
        st = lib().kda_prefill(*args, ws, ws_bytes, _stream_handle(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_prefill_recurrent" if recurrent else "kda_prefill")
    return out, final_state


def prefill_noalloc(q, k, v, log_alpha, beta, cu_seqlens, init_state=None, *, out, final_state=None,
                    lower_bound: float = -5.0, scale: float = 1.0, stream=None):
    """``kda_prefill_noalloc``: kda_prefill with the library's own scratch instead of a workspace,
    for callers that cannot allocate device memory (the caller still provides ``out`` and, if
    wanted, ``final_state``; nothing is allocated here either)."""
    T, H, d_k = q.shape
    d_v = v.shape[-1]
    N = cu_seqlens.shape[0] - 1
    _check_cuda(q, k, v, log_alpha, beta, cu_seqlens, init_state, out, final_state)
    st = lib().kda_prefill_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(cu_seqlens), N, T,
                                   H, d_k, d_v, _io_dtype(q.dtype), _io_dtype(out.dtype), float(lower_bound),
                                   float(scale), _ptr(init_state), _ptr(out), _ptr(final_state),
                                   _stream_handle(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_prefill_noalloc")
    return out, final_state


def prefill_gated(q, k, v, z, A_log, beta, cu_seqlens, init_state=None, *, out=None, final_state=None,
                  out_dtype=torch.float32, g_min: float = -5.0, scale: float = 1.0, stream=None,
                  recurrent: bool = False, want_final: bool = True):
    """KDA prefill with the gated log-decay g = g_min * Sigmoid(e^{A_h} z) (``kda_prefill_gated``).

    z [T, H, d_k] in the dtype of q/k/v; A_log [H] float32; the rest as in ``prefill``.
    ``recurrent=True`` forces the fp32 token-recurrent kernel (``kda_prefill_gated_recurrent``).
    """
    T, H, d_k = q.shape
    d_v = v.shape[-1]
    N = cu_seqlens.shape[0] - 1
    dt = _io_dtype(q.dtype)
    if k.dtype != q.dtype or v.dtype != q.dtype or z.dtype != q.dtype:
        raise TypeError("q, k, v and z must share one dtype")
    if A_log.dtype != torch.float32 or beta.dtype != torch.float32:
        raise TypeError("A_log and beta must be float32")
    if cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    if out is None:
        out = torch.empty((T, H, d_v), dtype=out_dtype, device=q.device)
    odt = _io_dtype(out.dtype)
    if final_state is None and want_final:
        final_state = torch.empty((N, H, d_k, d_v), dtype=torch.float32, device=q.device)
    _check_cuda(q, k, v, z, A_log, beta, cu_seqlens, init_state, out, final_state)
    fn = lib().kda_prefill_gated_recurrent if recurrent else lib().kda_prefill_gated
    st = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(A_log), _ptr(beta), _ptr(cu_seqlens), N, T, H, d_k, d_v, dt,
            odt, float(g_min), float(scale), _ptr(init_state), _ptr(out), _ptr(final_state), _stream_handle(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_prefill_gated_recurrent" if recurrent else "kda_prefill_gated")
    return out, final_state


def _decay_fields(q, log_alpha, lower_bound, z, A_log, g_min, unbounded=False):
    """(decay_form, decay tensor, A_log, bound) for exactly one of log_alpha or (z, A_log); with
    ``unbounded`` the logits go through the unbounded map g = -e^{A_h} Softplus(z)."""
    if (log_alpha is None) == (z is None):
        raise ValueError("pass exactly one of log_alpha (clamped form) or z with A_log (gated form)")
    if log_alpha is not None:
        if A_log is not None:
            raise ValueError("A_log belongs to the gated form (z)")
        if log_alpha.dtype != torch.float32:
            raise TypeError("log_alpha must be float32")
        return KDA_DECAY_CLAMPED, log_alpha, None, float(lower_bound)
    if A_log is None or A_log.dtype != torch.float32:
        raise TypeError("the gated form needs A_log [H] float32")
    if z.dtype != q.dtype:
        raise TypeError("z must have the dtype of q")
    return (KDA_DECAY_UNBOUNDED if unbounded else KDA_DECAY_GATED), z, A_log, float(g_min)


def prefill_ex(q, k, v, beta, cu_seqlens, *, log_alpha=None, lower_bound: float = -5.0, z=None, A_log=None,
               g_min: float = -5.0, init_state=None, out_gate=None, norm_weight=None, norm_eps: float = 1e-6,
               out=None, final_state=None, out_dtype=torch.float32, scale: float = 1.0, stream=None,
               recurrent: bool = False, want_final: bool = True, unbounded: bool = False, workspace="auto"):
    """Prefill through the parameter block (``kda_prefill_ex``): the clamped (``log_alpha``) or
    gated (``z``, ``A_log``) log-decay, and optionally the output gate with head-wise RMSNorm,
    ``out = Sigmoid(out_gate) * norm_weight * o / sqrt(mean(o^2) + norm_eps)`` per token and head.
    ``unbounded=True`` (with z, A_log) takes the earlier models' map g = -e^{A_h} Softplus(z)
    (chunked kernel for bf16 with d = 128, else the token-recurrent one).
    out_gate [T, H, d_v] in the dtype of q; norm_weight [d_v] float32 or None (ones).
    Returns (out, final_state or None)."""
    T, H, d_k = q.shape
    d_v = v.shape[-1]
    N = cu_seqlens.shape[0] - 1
    form, decay, A, bound = _decay_fields(q, log_alpha, lower_bound, z, A_log, g_min, unbounded)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    if out_gate is not None and out_gate.dtype != q.dtype:
        raise TypeError("out_gate must have the dtype of q")
    if norm_weight is not None and norm_weight.dtype != torch.float32:
        raise TypeError("norm_weight must be float32")
    if beta.dtype != torch.float32 or cu_seqlens.dtype != torch.int32:
        raise TypeError("beta must be float32 and cu_seqlens int32")
    if out is None:
        out = torch.empty((T, H, d_v), dtype=out_dtype, device=q.device)
    if final_state is None and want_final:
        final_state = torch.empty((N, H, d_k, d_v), dtype=torch.float32, device=q.device)
    _check_cuda(q, k, v, decay, A, beta, cu_seqlens, init_state, out_gate, norm_weight, out, final_state)
    ws, ws_bytes = _workspace(None if recurrent else workspace, T, N, H, d_k, d_v, q.device)
    p = PrefillParams(struct_size=ctypes.sizeof(PrefillParams), in_dtype=_io_dtype(q.dtype),
                      out_dtype=_io_dtype(out.dtype), decay_form=form, num_seqs=N, H=H, d_k=d_k, d_v=d_v,
                      total_tokens=T, q=q.data_ptr(), k=k.data_ptr(), v=v.data_ptr(), decay=decay.data_ptr(),
                      A_log=None if A is None else A.data_ptr(), beta=beta.data_ptr(),
                      cu_seqlens=cu_seqlens.data_ptr(),
                      init_state=None if init_state is None else init_state.data_ptr(),
                      out_gate=None if out_gate is None else out_gate.data_ptr(),
                      norm_weight=None if norm_weight is None else norm_weight.data_ptr(), out=out.data_ptr(),
                      final_state=None if final_state is None else final_state.data_ptr(), decay_bound=bound,
                      scale=float(scale), norm_eps=float(norm_eps), force_recurrent=int(bool(recurrent)),
                      workspace=ws, workspace_bytes=ws_bytes)
    st = lib().kda_prefill_ex(ctypes.byref(p), _stream_handle(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_prefill_ex")
    return out, final_state


def decode_ex(q, k, v, beta, state, *, log_alpha=None, lower_bound: float = -5.0, z=None, A_log=None,
              g_min: float = -5.0, out_gate=None, norm_weight=None, norm_eps: float = 1e-6, conv_weight=None,
              conv_state=None, l2_eps: float = 1e-6, out=None, out_dtype=torch.float32, scale: float = 1.0,
              stream=None, unbounded: bool = False):
    """One decode step through the parameter block (``kda_decode_ex``); ``state`` is updated in
    place. Decay and output-gate options as in ``prefill_ex``. With ``conv_state`` [B, H, 3,
    2 d_k + d_v] (dtype of q; shifted in place) and ``conv_weight`` [H, 2 d_k + d_v, 4] float32,
    q, k, v are the raw projections and pass the prologue of ``prologue`` first.
    Returns out [B, H, d_v]."""
    B, H, d_k = q.shape
    d_v = v.shape[-1]
    form, decay, A, bound = _decay_fields(q, log_alpha, lower_bound, z, A_log, g_min, unbounded)
    if out_gate is not None and out_gate.dtype != q.dtype:
        raise TypeError("out_gate must have the dtype of q")
    if out is None:
        out = torch.empty((B, H, d_v), dtype=out_dtype, device=q.device)
    _check_cuda(q, k, v, decay, A, beta, state, out_gate, norm_weight, conv_weight, conv_state, out)
    if conv_state is not None and conv_state.dtype != q.dtype:
        raise TypeError("conv_state must have the dtype of q")
    p = DecodeParams(struct_size=ctypes.sizeof(DecodeParams), in_dtype=_io_dtype(q.dtype),
                     out_dtype=_io_dtype(out.dtype), decay_form=form, B=B, H=H, d_k=d_k, d_v=d_v, q=q.data_ptr(),
                     k=k.data_ptr(), v=v.data_ptr(), decay=decay.data_ptr(),
                     A_log=None if A is None else A.data_ptr(), beta=beta.data_ptr(), state=state.data_ptr(),
                     out_gate=None if out_gate is None else out_gate.data_ptr(),
                     norm_weight=None if norm_weight is None else norm_weight.data_ptr(), out=out.data_ptr(),
                     conv_weight=None if conv_weight is None else conv_weight.data_ptr(),
                     conv_state=None if conv_state is None else conv_state.data_ptr(),
                     decay_bound=bound, scale=float(scale), norm_eps=float(norm_eps), l2_eps=float(l2_eps))
    st = lib().kda_decode_ex(ctypes.byref(p), _stream_handle(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_decode_ex")
    return out


def prologue(q_raw, k_raw, v_raw, conv_weight, cu_seqlens, conv_init=None, *, l2_eps: float = 1e-6, q=None,
             k=None, v=None, conv_final=None, want_final: bool = True, stream=None):
    """The input prologue (``kda_prologue``): 4-tap causal ShortConv per sequence, Swish, and the
    L2 norm of q and k. q_raw, k_raw [T, H, d_k], v_raw [T, H, d_v] (bf16 or fp32, one dtype);
    conv_weight [H, 2 d_k + d_v, 4] float32; conv_init [N, H, 3, 2 d_k + d_v] or None.
    Returns (q, k, v, conv_final or None), the inputs of ``prefill``."""
    T, H, d_k = q_raw.shape
    d_v = v_raw.shape[-1]
    N = cu_seqlens.shape[0] - 1
    dt = _io_dtype(q_raw.dtype)
    if k_raw.dtype != q_raw.dtype or v_raw.dtype != q_raw.dtype:
        raise TypeError("q, k and v must share one dtype")
    if conv_weight.dtype != torch.float32 or cu_seqlens.dtype != torch.int32:
        raise TypeError("conv_weight must be float32 and cu_seqlens int32")
    if conv_init is not None and conv_init.dtype != q_raw.dtype:
        raise TypeError("conv_init must have the dtype of q")
    q = torch.empty_like(q_raw) if q is None else q
    k = torch.empty_like(k_raw) if k is None else k
    v = torch.empty_like(v_raw) if v is None else v
    if conv_final is None and want_final:
        conv_final = torch.empty((N, H, 3, 2 * d_k + d_v), dtype=q_raw.dtype, device=q_raw.device)
    _check_cuda(q_raw, k_raw, v_raw, conv_weight, cu_seqlens, conv_init, q, k, v, conv_final)
    st = lib().kda_prologue(_ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(conv_weight), _ptr(cu_seqlens), N, T, H,
                            d_k, d_v, dt, _ptr(conv_init), float(l2_eps), _ptr(q), _ptr(k), _ptr(v),
                            _ptr(conv_final), _stream_handle(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_prologue")
    return q, k, v, conv_final


def decode_gated(q, k, v, z, A_log, beta, state, *, out=None, out_dtype=torch.float32, g_min: float = -5.0,
                 scale: float = 1.0, stream=None):
    """One decode step with the gated log-decay (``kda_decode_gated``); ``state`` is updated in place."""
    B, H, d_k = q.shape
    d_v = v.shape[-1]
    dt = _io_dtype(q.dtype)
    if z.dtype != q.dtype or A_log.dtype != torch.float32:
        raise TypeError("z must have the dtype of q, A_log must be float32")
    if out is None:
        out = torch.empty((B, H, d_v), dtype=out_dtype, device=q.device)
    odt = _io_dtype(out.dtype)
    _check_cuda(q, k, v, z, A_log, beta, state, out)
    st = lib().kda_decode_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(A_log), _ptr(beta), _ptr(state), _ptr(out),
                                B, H, d_k, d_v, dt, odt, float(g_min), float(scale), _stream_handle(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_decode_gated")
    return out


def decode(q, k, v, log_alpha, beta, state, *, out=None, out_dtype=torch.float32, lower_bound: float = -5.0,
           scale: float = 1.0, stream=None):
    """One KDA decode step (``kda_decode``); ``state`` [B, H, d_k, d_v] fp32 is updated in place.
    q, k [B, H, d_k], v [B, H, d_v]; log_alpha [B, H, d_k]; beta [B, H]. Returns out [B, H, d_v]."""
    B, H, d_k = q.shape
    d_v = v.shape[-1]
    dt = _io_dtype(q.dtype)
    if out is None:
        out = torch.empty((B, H, d_v), dtype=out_dtype, device=q.device)
    odt = _io_dtype(out.dtype)
    _check_cuda(q, k, v, log_alpha, beta, state, out)
    st = lib().kda_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(state), _ptr(out), B, H,
                          d_k, d_v, dt, odt, float(lower_bound), float(scale), _stream_handle(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_decode")
    return out


def check_device_error(stream=None):
    """Synchronise and raise if a kernel recorded a bounded-wait timeout or an input outside
    its range (``KdaError.status`` tells which)."""
    st = lib().kda_check_device_error(_stream_handle(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_check_device_error")


UMMA_FORMATS = {"f16": 0, "bf16": 1, "tf32": 2}


def selftest_umma(A, B, M, N, K, *, fmt="bf16", sw64=False, a_mn_major=False, b_mn_major=False, negate_a=False,
                  a_lbo=16, a_sbo=1024, b_lbo=16, b_sbo=1024, stream=None):
    """One tcgen05 MMA on the GPU (``kda_selftest_umma``); returns the raw [128, N] accumulator.
    A [M, K] and B [N, K] are rounded on the device to ``fmt`` (f16, bf16 or tf32)."""
    A32 = A.to(torch.float32).contiguous()
    B32 = B.to(torch.float32).contiguous()
    D = torch.full((128, N), float("nan"), dtype=torch.float32, device=A.device)
    status = torch.zeros(1, dtype=torch.int32, device=A.device)
    st = lib().kda_selftest_umma(_ptr(A32), _ptr(B32), _ptr(D), M, N, K, UMMA_FORMATS[fmt], int(sw64), int(a_mn_major),
                                 int(b_mn_major), int(negate_a), a_lbo, a_sbo, b_lbo, b_sbo, _ptr(status),
                                 _stream_handle(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_selftest_umma")
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise KdaError(KDA_ERR_TIMEOUT, "kda_selftest_umma")
    return D


def selftest_wait_timeout(stream=None):
    """Runs a bounded wait that is never satisfied (``kda_selftest_wait_timeout``); returns the
    kernel's status word (1 when the wait gave up). The device error word is left set for
    ``check_device_error`` to report."""
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = lib().kda_selftest_wait_timeout(_ptr(status), _stream_handle(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_selftest_wait_timeout")
    torch.cuda.synchronize()
    return int(status.item())


class HostPrefill:
    """End-to-end prefill from pinned HOST buffers, as an application calls it.

    Each ``__call__`` copies the inputs host -> device, runs ``kda_prefill`` and
    copies ``out`` and ``final_state`` back to pinned host memory, all on one
    stream, and waits for the result. Device staging buffers are allocated once.
    """

    def __init__(self, q, k, v, log_alpha, beta, cu_seqlens, init_state=None, device="cuda",
                 out_dtype=torch.float32):
        self.host_in = [t.pin_memory() if not t.is_pinned() else t
                        for t in (q, k, v, log_alpha, beta, cu_seqlens)]
        self.host_init = None if init_state is None else init_state.pin_memory()
        self.dev_in = [torch.empty_like(t, device=device) for t in self.host_in]
        self.dev_init = None if init_state is None else torch.empty_like(self.host_init, device=device)
        T, H, _ = q.shape
        N = cu_seqlens.shape[0] - 1
        self.dev_out = torch.empty((T, H, v.shape[-1]), dtype=out_dtype, device=device)
        self.dev_final = torch.empty((N, H, q.shape[-1], v.shape[-1]), dtype=torch.float32, device=device)
        self.host_out = torch.empty_like(self.dev_out, device="cpu").pin_memory()
        self.host_final = torch.empty_like(self.dev_final, device="cpu").pin_memory()

    @property
    def h2d_bytes(self) -> int:
        n = sum(t.numel() * t.element_size() for t in self.host_in)
        return n + (0 if self.host_init is None else self.host_init.numel() * 4)

    @property
    def d2h_bytes(self) -> int:
        return self.host_out.numel() * self.host_out.element_size() + self.host_final.numel() * 4

    def __call__(self, stream=None, sync: bool = True):
        stream = stream or torch.cuda.current_stream()
        with torch.cuda.stream(stream):
            for d, h in zip(self.dev_in, self.host_in):
                d.copy_(h, non_blocking=True)
            if self.dev_init is not None:
                self.dev_init.copy_(self.host_init, non_blocking=True)
            q, k, v, la, b, cu = self.dev_in
            prefill(q, k, v, la, b, cu, self.dev_init, out=self.dev_out, final_state=self.dev_final,
                    stream=stream)
            self.host_out.copy_(self.dev_out, non_blocking=True)
            self.host_final.copy_(self.dev_final, non_blocking=True)
        if sync:
            stream.synchronize()
        return self.host_out, self.host_final


class HostPrefillStream:
    """Prefill from pinned HOST buffers, streamed: step i's host-to-device copies, its kernel and
    its device-to-host copies run on three CUDA streams, so that step i+1's inputs travel while
    step i computes and step i-1's results come back.

    Every step still moves all its inputs to the device and all its outputs (``out`` and the
    final state) back to pinned host memory; two device staging sets and two host result sets
    alternate between steps. ``run(steps)`` enqueues the steps and waits for the last result.
    """

    def __init__(self, q, k, v, log_alpha, beta, cu_seqlens, init_state=None, device="cuda",
                 out_dtype=torch.float32):
        self.host_in = [t.pin_memory() if not t.is_pinned() else t
                        for t in (q, k, v, log_alpha, beta, cu_seqlens)]
        self.host_init = None if init_state is None else init_state.pin_memory()
        T, H, _ = q.shape
        N = cu_seqlens.shape[0] - 1
        self.dev_in = [[torch.empty_like(t, device=device) for t in self.host_in] for _ in range(2)]
        self.dev_init = [None if init_state is None else torch.empty_like(self.host_init, device=device)
                         for _ in range(2)]
        self.dev_out = [torch.empty((T, H, v.shape[-1]), dtype=out_dtype, device=device) for _ in range(2)]
        self.dev_final = [torch.empty((N, H, q.shape[-1], v.shape[-1]), dtype=torch.float32, device=device)
                          for _ in range(2)]
        self.host_out = [torch.empty_like(self.dev_out[0], device="cpu").pin_memory() for _ in range(2)]
        self.host_final = [torch.empty_like(self.dev_final[0], device="cpu").pin_memory() for _ in range(2)]
        self.s_in, self.s_run, self.s_back = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        self.ev_in = [torch.cuda.Event() for _ in range(2)]
        self.ev_run = [torch.cuda.Event() for _ in range(2)]
        self.ev_back = [torch.cuda.Event() for _ in range(2)]
        self.steps_done = 0

    @property
    def h2d_bytes(self) -> int:
        n = sum(t.numel() * t.element_size() for t in self.host_in)
        return n + (0 if self.host_init is None else self.host_init.numel() * 4)

    @property
    def d2h_bytes(self) -> int:
        return self.host_out[0].numel() * self.host_out[0].element_size() + self.host_final[0].numel() * 4

    def _in(self, i):
        b = i & 1
        with torch.cuda.stream(self.s_in):
            if i >= 2:
                self.s_in.wait_event(self.ev_run[b])  # step i-2's kernel has read this staging set
            for d, h in zip(self.dev_in[b], self.host_in):
                d.copy_(h, non_blocking=True)
            if self.dev_init[b] is not None:
                self.dev_init[b].copy_(self.host_init, non_blocking=True)
            self.ev_in[b].record(self.s_in)

    def _run(self, i):
        b = i & 1
        with torch.cuda.stream(self.s_run):
            self.s_run.wait_event(self.ev_in[b])
            if i >= 2:
                self.s_run.wait_event(self.ev_back[b])  # step i-2's results have left this set
            q, k, v, la, bt, cu = self.dev_in[b]
            prefill(q, k, v, la, bt, cu, self.dev_init[b], out=self.dev_out[b], final_state=self.dev_final[b],
                    stream=self.s_run)
            self.ev_run[b].record(self.s_run)

    def _back(self, i, stream):
        b = i & 1
        with torch.cuda.stream(stream):
            stream.wait_event(self.ev_run[b])
            self.host_out[b].copy_(self.dev_out[b], non_blocking=True)
            self.host_final[b].copy_(self.dev_final[b], non_blocking=True)
            self.ev_back[b].record(stream)

    def enqueue(self):
        """Enqueue one step (copies in, kernel, copies back) without waiting."""
        i = self.steps_done
        self._in(i)
        self._run(i)
        self._back(i, self.s_back)
        self.steps_done += 1

    def run(self, steps: int, duplex: bool = True):
        """Run ``steps`` streamed steps and return the last step's (out, final_state) on the host.
        ``duplex``: copies in and copies back on their own streams, so that both directions may
        run at once; otherwise one copy stream carries step i+1's inputs and then step i's
        results, so that the kernel still overlaps the copies but the two directions never do."""
        if duplex:
            for _ in range(steps):
                self.enqueue()
        elif steps > 0:
            i0 = self.steps_done
            self._in(i0)
            for n in range(steps):
                self._run(i0 + n)
                if n + 1 < steps:
                    self._in(i0 + n + 1)
                self._back(i0 + n, self.s_in)
            self.steps_done = i0 + steps
        b = (self.steps_done - 1) & 1
        self.ev_back[b].synchronize()
        return self.host_out[b], self.host_final[b]
