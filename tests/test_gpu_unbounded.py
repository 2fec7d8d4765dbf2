"""The unbounded log-decay of the earlier models, g = -e^{A_h} Softplus(z) (Kimi K3 --
Architecture Notes, section 1.2, the GDN / Mamba-2 / Kimi Linear row of the mapping table),
in prefill (bf16 requests with d = 128 take the chunked kernel, the others the
token-recurrent one) and in decode, against the fp64 oracle; decays far beyond -5 per step
are part of the cases. The chunked kernel's own cases are in test_gpu_unbounded_chunked.py."""

import numpy as np
import pytest
import torch

from helpers import TOL_BF16, TOL_F32, cpu, gated_output_err, rel_max_err
from kimi_delta_attention_02_gb300 import binding, workloads
from oracle import kda_recurrent_unbounded, output_gate_rmsnorm

pytestmark = pytest.mark.gpu


def _oracle(case):
    return kda_recurrent_unbounded(cpu(case.q), cpu(case.k), cpu(case.v), cpu(case.z), cpu(case.A_log),
                                   cpu(case.beta), cpu(case.cu_seqlens).long().numpy(),
                                   init_state=cpu(case.init_state))


def _run(case, **kw):
    out, fin = binding.prefill_ex(case.q, case.k, case.v, case.beta, case.cu_seqlens, z=case.z, A_log=case.A_log,
                                  init_state=case.init_state, unbounded=True, **kw)
    binding.check_device_error()
    return out, fin


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("lengths", [[1], [40], [0, 33, 5, 70]])
def test_prefill(lengths, dtype):
    case = workloads.make_prefill(lengths, H=3, dtype=dtype, device="cuda", seed=50 + sum(lengths), gated=True)
    out, fin = _run(case)
    o_ref, f_ref = _oracle(case)
    tol = TOL_BF16 if dtype == torch.bfloat16 else TOL_F32
    assert rel_max_err(out, o_ref) <= tol and rel_max_err(fin, f_ref) <= tol


def test_steep_decay_beyond_the_bound():
    """Logits of +40 at A_h = ln 2: g = -80 per step (alpha = e^-80), far below the -5 bound."""
    case = workloads.make_prefill([37], H=2, dtype=torch.float32, device="cuda", seed=51, gated=True)
    case.z[:, :, ::3] = 40.0
    case.A_log[:] = float(np.log(2.0))
    out, fin = _run(case)
    o_ref, f_ref = _oracle(case)
    assert rel_max_err(out, o_ref) <= TOL_F32 and rel_max_err(fin, f_ref) <= TOL_F32


def test_with_output_gate():
    case = workloads.make_prefill([50, 9], H=2, device="cuda", seed=53, gated=True, out_gate=True)
    out, fin = _run(case, out_gate=case.out_gate, norm_weight=case.norm_weight, norm_eps=1e-6)
    o_ref, f_ref = _oracle(case)
    y_ref = output_gate_rmsnorm(o_ref, cpu(case.out_gate), cpu(case.norm_weight), 1e-6)
    assert gated_output_err(out, y_ref, o_ref) <= TOL_BF16 and rel_max_err(fin, f_ref) <= TOL_BF16


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode(dtype):
    B, H = 5, 4
    st0 = workloads.make_decode_state(B, H, device="cuda", seed=54)
    step = workloads.make_decode_step(0, B, H, dtype=dtype, device="cuda", seed=54, gated=True)
    state = st0.clone()
    out = binding.decode_ex(step.q, step.k, step.v, step.beta, state, z=step.z, A_log=step.A_log, unbounded=True)
    binding.check_device_error()
    cu = np.arange(B + 1)
    o_ref, f_ref = kda_recurrent_unbounded(cpu(step.q), cpu(step.k), cpu(step.v), cpu(step.z), cpu(step.A_log),
                                           cpu(step.beta), cu, init_state=cpu(st0))
    tol = TOL_BF16 if dtype == torch.bfloat16 else TOL_F32
    assert rel_max_err(out, o_ref) <= tol and rel_max_err(state, f_ref) <= tol
