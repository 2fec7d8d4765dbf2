"""The output gate with head-wise RMSNorm (Kimi K3 -- Architecture Notes, section 1.3),
fused into the chunked prefill, the token-recurrent prefill and decode, against the
fp64 oracle: the recurrence, then Sigmoid(r) * w * o / sqrt(mean(o^2) + eps) per
token and head. Cases span several chunks and ragged tails, both decay forms, both
output dtypes, with and without the weight, and the K3-shaped layer in full."""

import numpy as np
import pytest
import torch

from helpers import TOL_BF16, TOL_F32, cpu, gated_output_err, oracle_prefill_out_gate, rel_max_err
from kimi_delta_attention_02_gb300 import binding, workloads
from oracle import kda_recurrent, kda_recurrent_gated, output_gate_rmsnorm

pytestmark = pytest.mark.gpu

EPS = 1e-6


def _run(case, *, recurrent=False, out_dtype=torch.float32, weight=True, eps=EPS, scale=1.0):
    kw = dict(z=case.z, A_log=case.A_log) if case.z is not None else dict(log_alpha=case.log_alpha)
    out, fin = binding.prefill_ex(case.q, case.k, case.v, case.beta, case.cu_seqlens, init_state=case.init_state,
                                  out_gate=case.out_gate, norm_weight=case.norm_weight if weight else None,
                                  norm_eps=eps, out_dtype=out_dtype, recurrent=recurrent, scale=scale, **kw)
    binding.check_device_error()
    return out, fin


def _check(case, tol, **kw):
    out, fin = _run(case, **kw)
    y_ref, f_ref, o_ref = oracle_prefill_out_gate(case, eps=kw.get("eps", EPS), scale=kw.get("scale", 1.0),
                                                  weight=kw.get("weight", True))
    e_y = gated_output_err(out, y_ref, o_ref, bf16_out=kw.get("out_dtype") == torch.bfloat16)
    e_f = rel_max_err(fin, f_ref)
    assert e_y <= tol and e_f <= tol, (e_y, e_f)
    return out


@pytest.mark.parametrize("T", [1, 17, 32, 33, 70, 96, 100, 257])
@pytest.mark.parametrize("gated", [False, True])
def test_chunked_lengths(T, gated):
    case = workloads.make_prefill([T], H=3, device="cuda", seed=40 + T, gated=gated, out_gate=True)
    _check(case, TOL_BF16)


def test_chunked_varlen_bf16_out_no_weight():
    case = workloads.make_prefill([0, 5, 64, 0, 131, 32], H=4, device="cuda", seed=41, out_gate=True)
    out = _check(case, TOL_BF16, out_dtype=torch.bfloat16, weight=False)
    assert out.dtype == torch.bfloat16


def test_chunked_scale_and_large_eps():
    """scale multiplies o before the norm; a large eps makes the norm see it."""
    case = workloads.make_prefill([77], H=2, device="cuda", seed=42, out_gate=True)
    _check(case, TOL_BF16, scale=0.25, eps=0.5)


@pytest.mark.parametrize("d_v", [128, 64, 100])
def test_recurrent_fp32(d_v):
    case = workloads.make_prefill([9, 40], H=2, d_k=96, d_v=d_v, dtype=torch.float32, device="cuda", seed=43,
                                  out_gate=True)
    _check(case, TOL_F32, recurrent=True)


def test_recurrent_fp32_unscaled_metric_wide_row_norms():
    """The output gate checked element by element with the plain metric max|dy| / rms(y), with no
    per-row weighting: q rows scaled by 10^u, u uniform in [-3, 1], give read-out rows whose norms
    span four decades, so an error confined to small-norm rows in the kernel's gate arithmetic
    (the RMS, the reciprocal square root, eps) shows up unscaled here."""
    case = workloads.make_prefill([9, 40], H=2, d_k=96, d_v=128, dtype=torch.float32, device="cuda", seed=47,
                                  out_gate=True)
    g = torch.Generator(device="cpu").manual_seed(47)
    s = 10.0 ** (4.0 * torch.rand(case.q.shape[:2], generator=g) - 3.0)
    case.q.mul_(s.to(case.q.device)[..., None])
    out, fin = _run(case, recurrent=True)
    y_ref, f_ref, o_ref = oracle_prefill_out_gate(case)
    row = np.sqrt((o_ref ** 2).mean(-1))
    assert row.max() / row.min() > 1e3
    assert rel_max_err(out, y_ref) <= TOL_F32 and rel_max_err(fin, f_ref) <= TOL_F32


def test_recurrent_matches_chunked():
    case = workloads.make_prefill([70, 3], H=2, device="cuda", seed=44, gated=True, out_gate=True)
    a, fa = _run(case)
    b, fb = _run(case, recurrent=True)
    _, _, o_ref = oracle_prefill_out_gate(case)
    assert gated_output_err(a, cpu(b).double().numpy(), o_ref) <= TOL_BF16


def test_plain_read_out_unchanged_by_parameter_block():
    """Without out_gate the parameter block gives exactly the plain entry point's results."""
    case = workloads.make_prefill([45], H=2, device="cuda", seed=45)
    a, fa = binding.prefill(case.q, case.k, case.v, case.log_alpha, case.beta, case.cu_seqlens, case.init_state)
    b, fb = binding.prefill_ex(case.q, case.k, case.v, case.beta, case.cu_seqlens, log_alpha=case.log_alpha,
                               init_state=case.init_state)
    assert torch.equal(a, b) and torch.equal(fa, fb)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_k3_layer_full_compare(out_dtype):
    """T=4096, H=96, gated decay, output gate: every output and state."""
    case = workloads.prefill_workload("prefill_k3_outgate_T4096_H96", device="cuda")
    _check(case, TOL_BF16, out_dtype=out_dtype)


@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode(gated, dtype):
    B, H = 5, 3
    state0 = workloads.make_decode_state(B, H, device="cuda", seed=46)
    st = workloads.make_decode_step(0, B, H, dtype=dtype, device="cuda", seed=46, gated=gated, out_gate=True)
    state = state0.clone()
    kw = dict(z=st.z, A_log=st.A_log) if gated else dict(log_alpha=st.log_alpha)
    out = binding.decode_ex(st.q, st.k, st.v, st.beta, state, out_gate=st.out_gate, norm_weight=st.norm_weight,
                            norm_eps=EPS, **kw)
    binding.check_device_error()
    cu = np.arange(B + 1)
    tok = lambda t: cpu(t)  # [B, H, d]: one token per sequence, packed token-major
    if gated:
        o, f = kda_recurrent_gated(tok(st.q), tok(st.k), tok(st.v), tok(st.z), cpu(st.A_log), cpu(st.beta), cu,
                                   init_state=cpu(state0))
    else:
        o, f = kda_recurrent(tok(st.q), tok(st.k), tok(st.v), tok(st.log_alpha), cpu(st.beta), cu,
                             init_state=cpu(state0))
    y = output_gate_rmsnorm(o, cpu(st.out_gate), cpu(st.norm_weight), EPS)
    tol = TOL_BF16 if dtype == torch.bfloat16 else TOL_F32
    assert gated_output_err(out, y, o) <= tol and rel_max_err(state, f) <= tol


def test_long_context_sampled_heads():
    """T = 2^20, H = 32 (the long-context shape) with the gated decay and the output gate: two
    seeded heads compared in full (heads are independent chains)."""
    case = workloads.make_prefill([1 << 20], H=32, device="cuda", seed=0, init_std=None, gated=True, out_gate=True)
    out, fin = _run(case, out_dtype=torch.bfloat16)
    heads = workloads.sampled_heads(32, 2, seed=1)
    sel = lambda t: t[:, heads].contiguous().cpu()
    o_ref, f_ref = kda_recurrent_gated(sel(case.q), sel(case.k), sel(case.v), sel(case.z), case.A_log[heads].cpu(),
                                       sel(case.beta), cpu(case.cu_seqlens).long().numpy())
    y_ref = output_gate_rmsnorm(o_ref, sel(case.out_gate), cpu(case.norm_weight), EPS)
    e_y = gated_output_err(out[:, heads], y_ref, o_ref, bf16_out=True)
    assert e_y <= TOL_BF16 and rel_max_err(fin[:, heads], f_ref) <= TOL_BF16, e_y
