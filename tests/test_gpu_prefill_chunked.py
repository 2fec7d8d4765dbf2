"""The tensor-core chunked prefill kernel (bf16 q/k/v, d = 128) against the fp64 oracle.

Every graded workload shape runs here in the launch configuration bench.py
times: the K3-shaped layer is compared in full; the varlen and 1M-token
workloads on seeded head samples (heads are independent chains, so a sampled
head's outputs and final state are exact oracle targets)."""

import os

import numpy as np
import pytest
import torch

from helpers import TOL_BF16, oracle_prefill, rel_max_err
from kimi_delta_attention_02_gb300 import binding, workloads
from oracle import kda_recurrent

pytestmark = pytest.mark.gpu


def _run(case, **kw):
    out, fin = binding.prefill(case.q, case.k, case.v, case.log_alpha, case.beta, case.cu_seqlens, case.init_state,
                               **kw)
    binding.check_device_error()
    return out, fin


def _oracle_heads(case, heads, threads=None):
    """Oracle on a subset of heads (each head of each sequence is an independent chain)."""
    sel = lambda t: t[:, heads].contiguous().cpu()
    init = None if case.init_state is None else case.init_state[:, heads].contiguous().cpu()
    return kda_recurrent(sel(case.q), sel(case.k), sel(case.v), sel(case.log_alpha), sel(case.beta),
                         case.cu_seqlens.cpu().long().numpy(), init_state=init,
                         num_threads=threads or os.cpu_count())


def _check(case, heads=None, tol=TOL_BF16):
    out, fin = _run(case)
    if heads is None:
        o_ref, f_ref = oracle_prefill(case)
        o, f = out, fin
    else:
        o_ref, f_ref = _oracle_heads(case, heads)
        o, f = out[:, heads], fin[:, heads]
    e_o, e_f = rel_max_err(o, o_ref), rel_max_err(f, f_ref)
    assert e_o <= tol and e_f <= tol, (e_o, e_f)
    return e_o, e_f


@pytest.mark.parametrize("T", [1, 15, 16, 17, 31, 32, 33, 63, 64, 65, 130, 1000])
def test_single_sequence_lengths(T):
    case = workloads.make_prefill([T], H=2, device="cuda", seed=T)
    _check(case)


def test_varlen_edge_lengths():
    case = workloads.make_prefill([0, 1, 31, 32, 33, 0, 200, 127], H=3, device="cuda", seed=11)
    out, fin = _run(case)
    assert torch.equal(fin[0], case.init_state[0]) and torch.equal(fin[5], case.init_state[5])
    _check(case)


def test_zero_initial_state_and_strong_forgetting():
    case = workloads.make_prefill([777], H=4, device="cuda", seed=12, init_std=None, log_alpha_mode="split")
    _check(case)


def test_lower_bound_at_minus_five_is_exact_clamp():
    """Every log-decay far below the bound: all retention factors equal e^-5 (the
    largest 16-token rescaling, e^80)."""
    case = workloads.make_prefill([256], H=2, device="cuda", seed=13)
    case.log_alpha.fill_(-30.0)
    _check(case)


def test_small_growth_is_computed_exactly():
    """Clamped log-decays up to +1/3 (retention factors above one) stay inside the chunked
    kernel's range: no status, and the oracle's results."""
    case = workloads.make_prefill([200], H=2, device="cuda", seed=18)
    case.log_alpha[20:51, 0, 5] = 0.25  # one key channel grows e^0.25 per token over 31 tokens (e^7.75)
    case.log_alpha[40:60, 1, :8] = 0.33  # eight channels at the edge of the range for 20 tokens
    _check(case)


def test_range_guard_reports_growth_beyond_the_envelope():
    """A clamped log-decay of +6 (alpha = e^6, far outside the method's (0, 1]) would overflow
    the chunked kernel's rescaled operands: the kernel reports KDA_ERR_RANGE through the device
    error word instead of returning silent Inf/NaN, and the token-recurrent kernel, which takes
    any finite log-decay, still matches the oracle on the same input."""
    case = workloads.make_prefill([96], H=2, device="cuda", seed=19)
    case.log_alpha[10:13, 1, 7] = 6.0
    binding.prefill(case.q, case.k, case.v, case.log_alpha, case.beta, case.cu_seqlens, case.init_state)
    with pytest.raises(binding.KdaError) as err:
        binding.check_device_error()
    assert err.value.status == binding.KDA_ERR_RANGE
    binding.check_device_error()  # the word was cleared by the check that reported it
    o_r, f_r = _run(case, recurrent=True)
    o_ref, f_ref = oracle_prefill(case)
    assert rel_max_err(o_r, o_ref) <= TOL_BF16 and rel_max_err(f_r, f_ref) <= TOL_BF16


def test_no_decay_and_zero_beta():
    case = workloads.make_prefill([190], H=2, device="cuda", seed=14)
    case.log_alpha.zero_()
    _check(case)
    case.beta.zero_()
    out, fin = _run(case)
    assert torch.equal(fin, case.init_state)  # alpha = 1, beta = 0: the state is untouched


def test_matches_recurrent_kernel_and_is_deterministic():
    case = workloads.make_prefill([1000, 333], H=4, device="cuda", seed=15)
    o1, f1 = _run(case)
    o2, f2 = _run(case)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)
    o_r, f_r = _run(case, recurrent=True)
    assert rel_max_err(o1, o_r.double().cpu().numpy()) < TOL_BF16
    assert rel_max_err(f1, f_r.double().cpu().numpy()) < TOL_BF16


def test_in_place_state_and_resume():
    case = workloads.make_prefill([300], H=2, device="cuda", seed=16)
    out, fin = _run(case)
    dev = case.q.device
    cut = 128
    cu1 = torch.tensor([0, cut], dtype=torch.int32, device=dev)
    cu2 = torch.tensor([0, 300 - cut], dtype=torch.int32, device=dev)
    sl = lambda t, a, b: t[a:b].contiguous()
    st = case.init_state.clone()
    o1, _ = binding.prefill(*(sl(t, 0, cut) for t in (case.q, case.k, case.v, case.log_alpha, case.beta)), cu1, st,
                            final_state=st)
    o2, _ = binding.prefill(*(sl(t, cut, 300) for t in (case.q, case.k, case.v, case.log_alpha, case.beta)), cu2,
                            st, final_state=st)
    assert rel_max_err(torch.cat([o1, o2]), out.double().cpu().numpy()) < 1e-5
    assert rel_max_err(st, fin.double().cpu().numpy()) < 1e-5


def test_bf16_output():
    case = workloads.make_prefill([500], H=2, device="cuda", seed=17)
    out, fin = _run(case, out_dtype=torch.bfloat16)
    o_ref, f_ref = oracle_prefill(case)
    o = out.double().cpu().numpy()
    rms = float((o_ref ** 2).mean() ** 0.5)
    assert (abs(o - o_ref) <= TOL_BF16 * rms + 2.0 ** -8 * abs(o_ref)).all()
    assert rel_max_err(fin, f_ref) < TOL_BF16


def test_k3_layer_full_compare():
    """B=1, T=4096, H=96, d=128, bf16, random fp32 initial state: every output and state."""
    case = workloads.prefill_workload("prefill_k3_T4096_H96", device="cuda")
    _check(case)


def test_varlen_workload_sampled_heads():
    """8 packed sequences of 1024..32768 tokens, H=96; heads 0..47 near the -5 bound,
    48..95 near zero decay. Checked on 4 seeded heads of each half."""
    case = workloads.prefill_workload("prefill_varlen8_H96", device="cuda")
    rng = np.random.default_rng(0)
    heads = sorted(rng.choice(48, 4, replace=False).tolist() + (48 + rng.choice(48, 4, replace=False)).tolist())
    _check(case, heads=heads)


def test_long_context_sampled_heads():
    """B=1, T=2^20, H=32, zero initial state; the seeded 4-head sample."""
    case = workloads.prefill_workload("prefill_long_T1M_H32", device="cuda")
    _check(case, heads=workloads.sampled_heads(32, 4, seed=0))


@pytest.mark.parametrize("streamed", [False, True, "half duplex"])
def test_host_buffer_prefill_matches_device_call(streamed):
    """The host-buffer paths (one step at a time, and streamed over two staging sets, with both
    copy directions on their own streams or on one) return exactly the device call's out and
    final state, at every step of a run; the streamed runs alternate the two modes."""
    case = workloads.make_prefill([40, 0, 97], H=4, device="cpu", seed=23)
    o_ref, f_ref = binding.prefill(*(t.cuda() for t in (case.q, case.k, case.v, case.log_alpha, case.beta,
                                                        case.cu_seqlens, case.init_state)))
    cls = binding.HostPrefillStream if streamed else binding.HostPrefill
    hp = cls(case.q, case.k, case.v, case.log_alpha, case.beta, case.cu_seqlens, case.init_state)
    for n, steps in enumerate((1, 1, 3, 2)):
        duplex = streamed is True if n % 2 == 0 else streamed is not True
        out, fin = hp.run(steps, duplex=duplex) if streamed else hp()
        assert out.device.type == "cpu" and fin.device.type == "cpu"
        assert torch.equal(out, o_ref.cpu()) and torch.equal(fin, f_ref.cpu())
    binding.check_device_error()
