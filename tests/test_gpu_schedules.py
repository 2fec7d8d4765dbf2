"""The chunked prefill's parallel schedules against the fp64 oracle: a single long sequence split
into segments (segment runs, an fp32 scan of the segments' affine maps S -> M S + B, then every
segment from its entering state), and packed sequences taken longest first. Both run only when
the caller passes the workspace kda_prefill_workspace_size asks for; without it one CTA per
(sequence, head) walks the chain."""

import numpy as np
import pytest
import torch

from helpers import TOL_BF16, gated_output_err, oracle_prefill, oracle_prefill_out_gate, rel_max_err
from kimi_delta_attention_02_gb300 import binding, workloads

pytestmark = pytest.mark.gpu


def _run(case, workspace, **kw):
    out, fin = binding.prefill(case.q, case.k, case.v, case.log_alpha, case.beta, case.cu_seqlens, case.init_state,
                               workspace=workspace, **kw)
    binding.check_device_error()
    return out, fin


@pytest.mark.parametrize("T,H", [(20000, 2), (9000, 3), (33000, 5)])
def test_segmented_single_sequence(T, H):
    """T = 20000 with 2 heads plans 4 segments (three-step scan), T = 9000 with 3 heads plans 2."""
    assert binding.workspace_size(T, 1, H) > 0
    case = workloads.make_prefill([T], H=H, device="cuda", seed=60 + H)
    out, fin = _run(case, "auto")
    o_ref, f_ref = oracle_prefill(case)
    e_o, e_f = rel_max_err(out, o_ref), rel_max_err(fin, f_ref)
    assert e_o <= TOL_BF16 and e_f <= TOL_BF16, (e_o, e_f)
    # against the one-CTA-per-head schedule of the same kernel
    out1, fin1 = _run(case, None)
    assert rel_max_err(out, out1.double().cpu().numpy()) <= TOL_BF16


def test_segmented_strong_forgetting_zero_init_and_in_place():
    """Half the heads near the -5 bound, half near zero decay, no initial state; then the same
    call continued in place (final_state = init_state) on a second sequence."""
    case = workloads.make_prefill([12345], H=4, device="cuda", seed=64, init_std=None, log_alpha_mode="split")
    out, fin = _run(case, "auto")
    o_ref, f_ref = oracle_prefill(case)
    assert rel_max_err(out, o_ref) <= TOL_BF16 and rel_max_err(fin, f_ref) <= TOL_BF16
    nxt = workloads.make_prefill([9999], H=4, device="cuda", seed=65)
    st = fin.clone()
    out2, _ = binding.prefill(nxt.q, nxt.k, nxt.v, nxt.log_alpha, nxt.beta, nxt.cu_seqlens, st, final_state=st)
    binding.check_device_error()
    nxt.init_state = fin
    o2_ref, f2_ref = oracle_prefill(nxt)
    assert rel_max_err(out2, o2_ref) <= TOL_BF16 and rel_max_err(st, f2_ref) <= TOL_BF16


def test_segmented_gated_decay_and_output_gate():
    """The gated decay map and the output gate (bf16 output) through the segmented schedule: the
    segment runs carry the state only, the output gate runs in the last pass."""
    case = workloads.make_prefill([10000], H=3, device="cuda", seed=66, gated=True, out_gate=True)
    out, fin = binding.prefill_ex(case.q, case.k, case.v, case.beta, case.cu_seqlens, z=case.z, A_log=case.A_log,
                                  init_state=case.init_state, out_gate=case.out_gate, norm_weight=case.norm_weight,
                                  out_dtype=torch.bfloat16, workspace="auto")
    binding.check_device_error()
    y_ref, f_ref, o_ref = oracle_prefill_out_gate(case)
    assert gated_output_err(out, y_ref, o_ref, bf16_out=True) <= TOL_BF16
    assert rel_max_err(fin, f_ref) <= TOL_BF16


def test_long_context_segmented_sampled_heads():
    """T = 2^20, H = 32 in the launch configuration the benchmark times (3 segments): the seeded
    4-head sample against the oracle."""
    case = workloads.prefill_workload("prefill_long_T1M_H32", device="cuda")
    assert binding.workspace_size(1 << 20, 1, 32) > 0
    out, fin = _run(case, "auto")
    heads = workloads.sampled_heads(32, 4, seed=0)
    sel = lambda t: t[:, heads].contiguous().cpu()
    from oracle import kda_recurrent
    o_ref, f_ref = kda_recurrent(sel(case.q), sel(case.k), sel(case.v), sel(case.log_alpha), sel(case.beta),
                                 case.cu_seqlens.cpu().long().numpy())
    e_o, e_f = rel_max_err(out[:, heads], o_ref), rel_max_err(fin[:, heads], f_ref)
    assert e_o <= TOL_BF16 and e_f <= TOL_BF16, (e_o, e_f)


def test_longest_first_order_is_bitwise_the_same():
    """Packed sequences in longest-first order: every chain runs the same arithmetic on another SM,
    so the results equal the in-order launch bit for bit."""
    lengths = [40, 3000, 0, 777, 65, 1, 2048, 129] * 3
    case = workloads.make_prefill(lengths, H=8, device="cuda", seed=67)
    assert binding.workspace_size(case.total_tokens, len(lengths), 8) > 0
    a, fa = _run(case, "auto")
    b, fb = _run(case, None)
    assert torch.equal(a, b) and torch.equal(fa, fb)
    o_ref, f_ref = oracle_prefill(case)
    assert rel_max_err(a, o_ref) <= TOL_BF16 and rel_max_err(fa, f_ref) <= TOL_BF16


def test_varlen_workload_ordered_sampled_heads():
    """The varlen workload (8 sequences, H = 96) in the benchmark's launch (longest first): four
    seeded heads of each decay half against the oracle."""
    case = workloads.prefill_workload("prefill_varlen8_H96", device="cuda")
    out, fin = _run(case, "auto")
    rng = np.random.default_rng(1)
    heads = sorted(rng.choice(48, 2, replace=False).tolist() + (48 + rng.choice(48, 2, replace=False)).tolist())
    sel = lambda t: t[:, heads].contiguous().cpu()
    from oracle import kda_recurrent
    o_ref, f_ref = kda_recurrent(sel(case.q), sel(case.k), sel(case.v), sel(case.log_alpha), sel(case.beta),
                                 case.cu_seqlens.cpu().long().numpy(), init_state=sel(case.init_state))
    assert rel_max_err(out[:, heads], o_ref) <= TOL_BF16 and rel_max_err(fin[:, heads], f_ref) <= TOL_BF16
