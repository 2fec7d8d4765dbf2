"""The unbounded log-decay g = -e^{A_h} Softplus(z) (Kimi K3 -- Architecture Notes, section 1.2,
the map of the earlier models) on the chunked tensor-core prefill, against the fp64 oracle.

Without a lower bound a channel's decay over a 16-token diagonal block of a chunk can pass
e^80; such a channel leaves the Gram for that block and its share is formed from position
pairs. The cases cover chunks without such a channel (the bounded path), chunks where every
channel has it, channels wide in only the first or only the second diagonal block, partial
chunks, several sequences, the output gate, and both output dtypes."""

import numpy as np
import pytest
import torch

from helpers import TOL_BF16, cpu, gated_output_err, rel_max_err
from kimi_delta_attention_02_gb300 import binding, workloads
from oracle import kda_recurrent_unbounded, output_gate_rmsnorm

pytestmark = pytest.mark.gpu


def _oracle(case):
    return kda_recurrent_unbounded(cpu(case.q), cpu(case.k), cpu(case.v), cpu(case.z), cpu(case.A_log),
                                   cpu(case.beta), cpu(case.cu_seqlens).long().numpy(),
                                   init_state=cpu(case.init_state), num_threads=8)


def _run(case, **kw):
    out, fin = binding.prefill_ex(case.q, case.k, case.v, case.beta, case.cu_seqlens, z=case.z, A_log=case.A_log,
                                  init_state=case.init_state, unbounded=True, **kw)
    binding.check_device_error()
    return out, fin


def _check(case, **kw):
    out, fin = _run(case, **kw)
    o_ref, f_ref = _oracle(case)
    e_o, e_f = rel_max_err(out, o_ref), rel_max_err(fin, f_ref)
    assert e_o <= TOL_BF16 and e_f <= TOL_BF16, (e_o, e_f)
    return out, fin


@pytest.mark.parametrize("lengths", [[1], [31], [32], [33], [100, 7, 64], [0, 129, 0, 16]])
def test_logit_distribution(lengths):
    """The gated workload's logits through the unbounded map (mostly chunks without wide channels)."""
    case = workloads.make_prefill(lengths, H=3, device="cuda", seed=300 + sum(lengths), gated=True)
    _check(case)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("lengths", [[37], [64, 45], [96]])
def test_steep_decay_every_third_channel(lengths, out_dtype):
    """Logits of +40 at A_h = ln 2 on every third channel: g = -80 per step there, so every
    chunk has wide channels in both diagonal blocks; the other channels keep the tensor cores."""
    case = workloads.make_prefill(lengths, H=2, device="cuda", seed=310 + sum(lengths), gated=True)
    case.z[:, :, ::3] = 40.0
    case.A_log[:] = float(np.log(2.0))
    out = torch.empty(case.v.shape, dtype=out_dtype, device="cuda")
    _check(case, out=out)


def test_every_channel_wide():
    case = workloads.make_prefill([70, 5], H=2, device="cuda", seed=320, gated=True)
    case.z[:] = 30.0
    case.A_log[:] = float(np.log(1.5))
    _check(case)


@pytest.mark.parametrize("block", [0, 1])
def test_one_diagonal_block_wide(block):
    """Steep decay on tokens of one 16-token half of each chunk only, in a few channels, so
    that a channel is wide in one diagonal block and on the tensor cores in the other."""
    case = workloads.make_prefill([96, 40], H=2, device="cuda", seed=330 + block, gated=True)
    t = torch.arange(case.z.shape[0], device="cuda")
    starts = case.cu_seqlens.long()
    pos = t - starts[torch.searchsorted(starts[1:], t, right=True)]  # position inside its sequence
    rows = ((pos % 32) // 16) == block
    sel = case.z[rows]
    sel[:, :, 5:40:7] = 25.0
    case.z[rows] = sel
    _check(case)


def test_occasional_wide_group():
    """A few isolated steep steps (+25 logits on single tokens of single channels): chunks
    switch between the bounded path and the position-pair path along the sequence."""
    case = workloads.make_prefill([300], H=4, device="cuda", seed=340, gated=True)
    g = torch.Generator().manual_seed(340)
    T, H, d = case.z.shape
    idx = torch.randint(0, T * H * d, (60,), generator=g)
    flat = case.z.view(-1)
    flat[idx.to("cuda")] = 25.0
    case.A_log[:] = float(np.log(3.0))
    _check(case)


def test_with_output_gate():
    case = workloads.make_prefill([50, 90], H=2, device="cuda", seed=350, gated=True, out_gate=True)
    case.z[:, :, ::5] = 40.0
    out, fin = _run(case, out_gate=case.out_gate, norm_weight=case.norm_weight, norm_eps=1e-6)
    o_ref, f_ref = _oracle(case)
    y_ref = output_gate_rmsnorm(o_ref, cpu(case.out_gate), cpu(case.norm_weight), 1e-6)
    assert gated_output_err(out, y_ref, o_ref) <= TOL_BF16 and rel_max_err(fin, f_ref) <= TOL_BF16


def test_agrees_with_token_recurrent_kernel():
    """The chunked result and the forced token-recurrent one agree to the bf16 tolerance."""
    case = workloads.make_prefill([65, 200], H=2, device="cuda", seed=360, gated=True)
    case.z[:, 1, ::4] = 35.0
    a, fa = _run(case)
    b, fb = _run(case, recurrent=True)
    assert rel_max_err(a, b.double().cpu().numpy()) <= TOL_BF16
    assert rel_max_err(fa, fb.double().cpu().numpy()) <= TOL_BF16


def test_long_sequence_heads():
    """T = 4096 at H = 4 with the gated workload's logits, full-size chunks throughout."""
    case = workloads.make_prefill([4096], H=4, device="cuda", seed=370, gated=True)
    _check(case)


def test_benchmark_workload_sampled_heads():
    """The benchmark's T=4096, H=96 logits through the unbounded map, in the launch `bench.py`
    times, checked on four heads: the one with the largest e^{A_h} (the most chunks with wide
    channels), the smallest, and two others."""
    case = workloads.prefill_workload("prefill_k3_gated_T4096_H96", device="cuda")
    out, fin = _run(case)
    A = case.A_log.cpu()
    heads = sorted({int(A.argmax()), int(A.argmin()), 17, 60})
    sel = lambda t: cpu(t[:, heads]).contiguous()
    o_ref, f_ref = kda_recurrent_unbounded(sel(case.q), sel(case.k), sel(case.v), sel(case.z), A[heads].contiguous(),
                                           sel(case.beta), cpu(case.cu_seqlens).long().numpy(),
                                           init_state=cpu(case.init_state[:, heads]).contiguous(), num_threads=4)
    e_o, e_f = rel_max_err(out[:, heads], o_ref), rel_max_err(fin[:, heads], f_ref)
    assert e_o <= TOL_BF16 and e_f <= TOL_BF16, (heads, e_o, e_f)
