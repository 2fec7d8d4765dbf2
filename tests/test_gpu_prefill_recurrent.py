"""The fp32 token-recurrent prefill kernel on the GPU against the fp64 oracle."""

import pytest
import torch

from helpers import TOL_F32, oracle_prefill, rel_max_err, tol_for
from kimi_delta_attention_02_gb300 import binding, workloads

pytestmark = pytest.mark.gpu


def _to(case, dev):
    for name in ("q", "k", "v", "log_alpha", "beta", "cu_seqlens", "init_state"):
        t = getattr(case, name)
        setattr(case, name, None if t is None else t.to(dev))
    return case


def _check(case, recurrent=True, **kw):
    out, fin = binding.prefill(case.q, case.k, case.v, case.log_alpha, case.beta, case.cu_seqlens,
                               case.init_state, recurrent=recurrent, **kw)
    binding.check_device_error()
    o_ref, f_ref = oracle_prefill(case, **{k: v for k, v in kw.items() if k in ("lower_bound", "scale")})
    tol = tol_for(case.q.dtype)
    e_o, e_f = rel_max_err(out, o_ref), rel_max_err(fin, f_ref)
    assert e_o <= tol and e_f <= tol, (e_o, e_f)
    return out, fin


def test_fp32_workload_through_kda_prefill():
    """fp32 everywhere, B=1, T=256, H=2, d=128, chunk-free, zero initial state (tolerance 1e-4)."""
    case = workloads.prefill_workload("prefill_f32_T256_H2", device="cuda")
    assert case.init_state is None
    _check(case, recurrent=False)


@pytest.mark.parametrize("d_k,d_v", [(16, 16), (32, 64), (64, 128), (100, 40), (128, 1)])
def test_fp32_odd_head_dims(d_k, d_v):
    case = workloads.make_prefill([37, 90], H=2, d_k=d_k, d_v=d_v, dtype=torch.float32, device="cuda", seed=2)
    _check(case)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_varlen_edge_lengths(dtype):
    """Empty, length-1, and lengths around the 64-token chunk boundary in one packed call."""
    case = workloads.make_prefill([0, 1, 63, 64, 65, 0, 200], H=3, dtype=dtype, device="cuda", seed=4)
    out, fin = _check(case)
    assert torch.equal(fin[0], case.init_state[0]) and torch.equal(fin[5], case.init_state[5])


def test_strong_forgetting_and_clamp():
    case = workloads.make_prefill([300], H=4, dtype=torch.float32, device="cuda", seed=5, log_alpha_mode="split")
    _check(case)


def test_scale_and_lower_bound_parameters():
    case = workloads.make_prefill([77], H=2, dtype=torch.float32, device="cuda", seed=6)
    _check(case, lower_bound=-2.0, scale=0.125)


def test_in_place_final_state_and_determinism():
    case = workloads.make_prefill([129, 5], H=2, dtype=torch.bfloat16, device="cuda", seed=7)
    o1, f1 = binding.prefill(case.q, case.k, case.v, case.log_alpha, case.beta, case.cu_seqlens, case.init_state,
                             recurrent=True)
    o2, f2 = binding.prefill(case.q, case.k, case.v, case.log_alpha, case.beta, case.cu_seqlens, case.init_state,
                             recurrent=True)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)
    st = case.init_state.clone()
    o3, _ = binding.prefill(case.q, case.k, case.v, case.log_alpha, case.beta, case.cu_seqlens, st,
                            final_state=st, recurrent=True)
    assert torch.equal(o3, o1) and torch.equal(st, f1)


def test_split_and_resume():
    case = workloads.make_prefill([211], H=2, dtype=torch.float32, device="cuda", seed=8)
    out, fin = binding.prefill(case.q, case.k, case.v, case.log_alpha, case.beta, case.cu_seqlens, case.init_state,
                               recurrent=True)
    cut = 100
    dev = case.q.device
    cu1 = torch.tensor([0, cut], dtype=torch.int32, device=dev)
    cu2 = torch.tensor([0, 211 - cut], dtype=torch.int32, device=dev)
    sl = lambda t, a, b: t[a:b].contiguous()
    o1, f1 = binding.prefill(*(sl(t, 0, cut) for t in (case.q, case.k, case.v, case.log_alpha, case.beta)), cu1,
                             case.init_state, recurrent=True)
    o2, f2 = binding.prefill(*(sl(t, cut, 211) for t in (case.q, case.k, case.v, case.log_alpha, case.beta)), cu2,
                             f1, recurrent=True)
    ref_o = out.double().cpu().numpy()
    assert rel_max_err(torch.cat([o1, o2]), ref_o) < 1e-5
    assert rel_max_err(f2, fin.double().cpu().numpy()) < 1e-5


def test_bf16_output_within_one_ulp():
    """bf16 outputs: the fp32 result rounded once, so each element is within the
    computation tolerance plus one bf16 rounding (2^-8 relative, conservatively)."""
    case = workloads.make_prefill([150, 70], H=2, dtype=torch.bfloat16, device="cuda", seed=3)
    out, fin = binding.prefill(case.q, case.k, case.v, case.log_alpha, case.beta, case.cu_seqlens, case.init_state,
                               out_dtype=torch.bfloat16, recurrent=True)
    o_ref, f_ref = oracle_prefill(case)
    o = out.double().cpu().numpy()
    rms = float((o_ref ** 2).mean() ** 0.5)
    assert (abs(o - o_ref) <= 1e-3 * rms + 2.0 ** -8 * abs(o_ref)).all()
    assert rel_max_err(fin, f_ref) < 1e-4
