"""The Python binding's host-side checks, run without a GPU. Every entry point refuses host
(CPU) tensors with an error instead of computing anything on the CPU: there is no fallback
path. The decay options and dtypes are validated before anything reaches the library."""

import pytest
import torch

from kimi_delta_attention_02_gb300 import binding as B
from kimi_delta_attention_02_gb300 import workloads

CUDA_ONLY = "contiguous CUDA tensors"


def _case(**kw):
    return workloads.make_prefill([40, 7], H=2, device="cpu", seed=3, **kw)


def test_prefill_entry_points_refuse_host_tensors():
    c = _case()
    with pytest.raises(ValueError, match=CUDA_ONLY):
        B.prefill(c.q, c.k, c.v, c.log_alpha, c.beta, c.cu_seqlens, c.init_state)
    with pytest.raises(ValueError, match=CUDA_ONLY):
        B.prefill(c.q, c.k, c.v, c.log_alpha, c.beta, c.cu_seqlens, c.init_state, recurrent=True)
    with pytest.raises(ValueError, match=CUDA_ONLY):
        B.prefill_noalloc(c.q, c.k, c.v, c.log_alpha, c.beta, c.cu_seqlens, c.init_state,
                          out=torch.empty(c.v.shape, dtype=torch.float32))
    g = _case(gated=True, out_gate=True)
    with pytest.raises(ValueError, match=CUDA_ONLY):
        B.prefill_gated(g.q, g.k, g.v, g.z, g.A_log, g.beta, g.cu_seqlens, g.init_state)
    for unbounded in (False, True):
        with pytest.raises(ValueError, match=CUDA_ONLY):
            B.prefill_ex(g.q, g.k, g.v, g.beta, g.cu_seqlens, z=g.z, A_log=g.A_log, init_state=g.init_state,
                         out_gate=g.out_gate, norm_weight=g.norm_weight, unbounded=unbounded)


def test_decode_entry_points_refuse_host_tensors():
    state = workloads.make_decode_state(2, 2, device="cpu", seed=1)
    st = workloads.make_decode_step(0, 2, 2, device="cpu", seed=1, gated=True)
    with pytest.raises(ValueError, match=CUDA_ONLY):
        B.decode(st.q, st.k, st.v, st.log_alpha, st.beta, state)
    with pytest.raises(ValueError, match=CUDA_ONLY):
        B.decode_gated(st.q, st.k, st.v, st.z, st.A_log, st.beta, state)
    with pytest.raises(ValueError, match=CUDA_ONLY):
        B.decode_ex(st.q, st.k, st.v, st.beta, state, z=st.z, A_log=st.A_log, unbounded=True)


def test_prologue_refuses_host_tensors():
    p = workloads.make_prologue([20, 3], H=2, device="cpu", seed=2)
    with pytest.raises(ValueError, match=CUDA_ONLY):
        B.prologue(p.q_raw, p.k_raw, p.v_raw, p.conv_weight, p.cu_seqlens, p.conv_init)


def test_prefill_ex_decay_options():
    c, g = _case(), _case(gated=True)
    common = (c.q, c.k, c.v, c.beta, c.cu_seqlens)
    with pytest.raises(ValueError, match="exactly one"):  # both forms at once
        B.prefill_ex(*common, log_alpha=c.log_alpha, z=g.z, A_log=g.A_log)
    with pytest.raises(ValueError, match="exactly one"):  # neither
        B.prefill_ex(*common)
    with pytest.raises(ValueError, match="A_log belongs"):
        B.prefill_ex(*common, log_alpha=c.log_alpha, A_log=g.A_log)
    with pytest.raises(TypeError, match="A_log"):  # the gated form without its per-head scale
        B.prefill_ex(*common, z=g.z)
    with pytest.raises(TypeError, match="log_alpha"):
        B.prefill_ex(*common, log_alpha=c.log_alpha.half())
    with pytest.raises(TypeError, match="z must"):
        B.prefill_ex(*common, z=g.z.float(), A_log=g.A_log)


def test_prefill_dtype_checks():
    c = _case()
    with pytest.raises(TypeError, match="one dtype"):
        B.prefill(c.q, c.k.float(), c.v, c.log_alpha, c.beta, c.cu_seqlens)
    with pytest.raises(TypeError, match="int32"):
        B.prefill(c.q, c.k, c.v, c.log_alpha, c.beta, c.cu_seqlens.long())
    with pytest.raises(TypeError, match="float32"):
        B.prefill(c.q, c.k, c.v, c.log_alpha.double(), c.beta, c.cu_seqlens)
