"""The gated log-decay g = g_min * Sigmoid(e^{A_h} z) (Kimi K3 -- Architecture
Notes, section 1.2, the K3 row of the mapping table) on the GPU against the
fp64 oracle: the chunked tensor-core kernel (bf16, d = 128, g_min >= -5), the
token-recurrent kernel (fp32 inputs, other head sizes, g_min < -5) and decode."""

import numpy as np
import pytest
import torch

from helpers import TOL_BF16, TOL_F32, oracle_prefill_gated, rel_max_err, tol_for
from kimi_delta_attention_02_gb300 import binding, workloads
from oracle import kda_recurrent_gated

pytestmark = pytest.mark.gpu


def _run(case, g_min=-5.0, **kw):
    out, fin = binding.prefill_gated(case.q, case.k, case.v, case.z, case.A_log, case.beta, case.cu_seqlens,
                                     case.init_state, g_min=g_min, **kw)
    binding.check_device_error()
    return out, fin


def _check(case, tol, g_min=-5.0, heads=None, **kw):
    out, fin = _run(case, g_min=g_min, **kw)
    o_ref, f_ref = oracle_prefill_gated(case, g_min=g_min, heads=heads)
    if heads is not None:
        out, fin = out[:, heads], fin[:, heads]
    e_o, e_f = rel_max_err(out, o_ref), rel_max_err(fin, f_ref)
    assert e_o <= tol and e_f <= tol, (e_o, e_f)
    return e_o, e_f


@pytest.mark.parametrize("T", [1, 17, 32, 33, 130, 1000])
def test_chunked_gated_lengths(T):
    case = workloads.make_prefill([T], H=2, device="cuda", seed=40 + T, gated=True)
    _check(case, TOL_BF16)


def test_chunked_gated_varlen_edges():
    case = workloads.make_prefill([0, 1, 31, 32, 33, 0, 200, 127], H=3, device="cuda", seed=41, gated=True)
    out, fin = _run(case)
    assert torch.equal(fin[0], case.init_state[0]) and torch.equal(fin[5], case.init_state[5])
    _check(case, TOL_BF16)


def test_chunked_gated_saturated_logits():
    """|e^{A_h} z| large: every step at the bound (g -> g_min, strongest decay) or at alpha = 1."""
    case = workloads.make_prefill([300], H=2, device="cuda", seed=42, gated=True)
    sign = torch.where(torch.rand(case.z.shape, device="cuda") > 0.5, 1.0, -1.0)
    case.z.copy_((60.0 * sign).to(case.z.dtype))
    _check(case, TOL_BF16)


def test_chunked_gated_k3_layer_full_compare():
    """B=1, T=4096, H=96, d=128, bf16 logits, random fp32 initial state: every output and state."""
    case = workloads.prefill_workload("prefill_k3_gated_T4096_H96", device="cuda")
    _check(case, TOL_BF16)


def test_chunked_gated_matches_recurrent_kernel():
    case = workloads.make_prefill([700, 333], H=4, device="cuda", seed=43, gated=True)
    o1, f1 = _run(case)
    o_r, f_r = _run(case, recurrent=True)
    assert rel_max_err(o1, o_r.double().cpu().numpy()) < TOL_BF16
    assert rel_max_err(f1, f_r.double().cpu().numpy()) < TOL_BF16


def test_recurrent_gated_fp32():
    case = workloads.make_prefill([256], H=2, dtype=torch.float32, device="cuda", seed=44, init_std=None, gated=True)
    _check(case, TOL_F32)


def test_recurrent_gated_odd_heads_and_low_bound():
    """d_k = 64, d_v = 32 in fp32, and a g_min of -8 on the bf16 path (below the chunked kernel's range)."""
    case = workloads.make_prefill([90, 40], H=2, d_k=64, d_v=32, dtype=torch.float32, device="cuda", seed=45,
                                  gated=True)
    _check(case, TOL_F32)
    case = workloads.make_prefill([150], H=2, device="cuda", seed=46, gated=True)
    _check(case, TOL_BF16, g_min=-8.0)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_gated(dtype):
    """Steps of kda_decode_gated on every (sequence, head) pair, replayed by the oracle as one
    sequence per pair."""
    dev = torch.device("cuda")
    B, H, steps = 5, 3, 6
    state0 = workloads.make_decode_state(B, H, device=dev, seed=3)
    state = state0.clone()
    seq = {name: [] for name in ("q", "k", "v", "z", "beta", "out")}
    A = None
    for s in range(steps):
        st = workloads.make_decode_step(s, B, H, dtype=dtype, device=dev, seed=3, gated=True)
        A = st.A_log
        out = binding.decode_gated(st.q, st.k, st.v, st.z, st.A_log, st.beta, state)
        for name in ("q", "k", "v", "z", "beta"):
            seq[name].append(getattr(st, name).cpu())
        seq["out"].append(out.cpu())
    binding.check_device_error()
    P = B * H
    # sequence (b, h) -> its steps in order; head h keeps its own A_h: lay pairs out as [steps, B, H]
    stack = lambda xs: torch.stack(xs, dim=0).permute(1, 0, 2, 3).reshape(B * steps, H, -1)
    beta = torch.stack(seq["beta"], dim=0).permute(1, 0, 2).reshape(B * steps, H)
    cu = np.arange(0, B * steps + 1, steps, dtype=np.int64)
    o_ref, f_ref = kda_recurrent_gated(stack(seq["q"]), stack(seq["k"]), stack(seq["v"]), stack(seq["z"]), A.cpu(),
                                       beta, cu, init_state=state0.cpu())
    tol = tol_for(dtype)
    e_o, e_f = rel_max_err(stack(seq["out"]), o_ref), rel_max_err(state, f_ref)
    assert e_o <= tol and e_f <= tol, (e_o, e_f)
