"""The input prologue (Kimi K3 -- Architecture Notes, section 1.1: ShortConv, Swish, the L2
norm of q and k) on the GPU against the fp64 oracle: the standalone prefill pass over packed
sequences (tiles that straddle sequences, sequences shorter than the window, empty ones,
with and without initial states) and the fused decode step with its convolution state.

Tolerances: a result in the workload dtype is within one rounding of the oracle (2^-8 of
|ref| for bf16, at most half a unit in the last place) plus 1e-5 of |ref| and 1e-6 of the
tensor's rms for the fp32 arithmetic (fp32 results: 1e-5 of |ref|); the
convolution states are raw inputs moved around, so they must match bit for bit."""

import numpy as np
import pytest
import torch

from helpers import TOL_BF16, TOL_F32, cpu, rel_max_err
from kimi_delta_attention_02_gb300 import binding, workloads
from oracle import kda_prologue, kda_recurrent

pytestmark = pytest.mark.gpu

EPS = 1e-6


def _close(gpu, ref, dtype):
    g = gpu.detach().double().cpu().numpy()
    rel = (2.0 ** -8 + 1e-5) if dtype == torch.bfloat16 else 1e-5
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    bad = np.abs(g - ref) > rel * np.abs(ref) + 1e-6 * rms
    assert not bad.any(), (int(bad.sum()), float(np.abs(g - ref).max()))


def _run(case, **kw):
    q, k, v, fin = binding.prologue(case.q_raw, case.k_raw, case.v_raw, case.conv_weight, case.cu_seqlens,
                                    case.conv_init, l2_eps=EPS, **kw)
    binding.check_device_error()
    return q, k, v, fin


def _check(case, dtype):
    q, k, v, fin = _run(case)
    qr, kr, vr, fr = kda_prologue(cpu(case.q_raw), cpu(case.k_raw), cpu(case.v_raw), cpu(case.conv_weight),
                                  cpu(case.cu_seqlens).long().numpy(), cpu(case.conv_init), eps=EPS)
    _close(q, qr, dtype)
    _close(k, kr, dtype)
    _close(v, vr, dtype)
    assert np.array_equal(fin.double().cpu().numpy(), fr)  # raw values moved: exact
    return q, k, v, fin


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("lengths", [[1], [2, 0, 3], [31, 1, 33, 2, 64], [100], [0, 5, 0]])
def test_prefill_pass(lengths, dtype):
    case = workloads.make_prologue(lengths, H=3, dtype=dtype, device="cuda", seed=len(lengths) + sum(lengths))
    _check(case, dtype)


def test_prefill_pass_zero_state_and_odd_sizes():
    case = workloads.make_prologue([7, 40, 1], H=2, d_k=64, d_v=100, dtype=torch.float32, device="cuda", seed=5,
                                   with_state=False)
    _check(case, torch.float32)


def test_prefill_pass_k3_layer():
    """T=4096, H=96: the K3-shaped layer's raw projections, every element."""
    case = workloads.make_prologue([4096], H=96, device="cuda", seed=0)
    _check(case, torch.bfloat16)


def test_prologue_then_prefill():
    """The prologue's outputs feed the chunked prefill; the oracle recurrence on the same bf16
    tensors agrees within the bf16-path tolerance."""
    case = workloads.make_prologue([70, 33], H=2, device="cuda", seed=6)
    q, k, v, _ = _check(case, torch.bfloat16)
    T, H = q.shape[:2]
    g = torch.Generator(device="cpu").manual_seed(1)
    la = (-torch.nn.functional.softplus(torch.randn((T, H, 128), generator=g))).cuda()
    beta = torch.sigmoid(torch.randn((T, H), generator=g)).cuda()
    out, fin = binding.prefill(q, k, v, la, beta, case.cu_seqlens)
    o_ref, f_ref = kda_recurrent(cpu(q), cpu(k), cpu(v), cpu(la), cpu(beta), cpu(case.cu_seqlens).long().numpy())
    assert rel_max_err(out, o_ref) <= TOL_BF16 and rel_max_err(fin, f_ref) <= TOL_BF16


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_step_with_conv_state(dtype):
    """One decode step on raw q, k, v: the conv state shifts in place, the step equals the
    oracle prologue (one token per sequence, the state before it) followed by the recurrence."""
    B, H = 6, 3
    st0 = workloads.make_decode_state(B, H, device="cuda", seed=7)
    cs0 = workloads.make_conv_state(B, H, dtype=dtype, device="cuda", seed=7)
    w = workloads.make_conv_weight(H, device="cuda", seed=7)
    step = workloads.make_decode_step(0, B, H, dtype=dtype, device="cuda", seed=8)
    g = torch.Generator(device="cpu").manual_seed(2)
    qr, kr, vr = (torch.randn(t.shape, generator=g).to(dtype).cuda() for t in (step.q, step.k, step.v))
    state, cs = st0.clone(), cs0.clone()
    out = binding.decode_ex(qr, kr, vr, step.beta, state, log_alpha=step.log_alpha, conv_weight=w, conv_state=cs,
                            l2_eps=EPS)
    binding.check_device_error()
    cu = np.arange(B + 1)
    q, k, v, fin = kda_prologue(cpu(qr), cpu(kr), cpu(vr), cpu(w), cu, cpu(cs0), eps=EPS)
    o_ref, f_ref = kda_recurrent(q, k, v, cpu(step.log_alpha), cpu(step.beta), cu, init_state=cpu(st0))
    assert np.array_equal(cs.double().cpu().numpy(), fin)
    tol = TOL_BF16 if dtype == torch.bfloat16 else TOL_F32
    assert rel_max_err(out, o_ref) <= tol and rel_max_err(state, f_ref) <= tol


def test_prefill_state_continues_into_decode():
    """The prologue's final conv state over tokens 0..T-1, handed to decode, gives token T the
    same processed inputs as a prologue pass over tokens 0..T."""
    H = 2

    def on_gpu(c):
        for name in ("q_raw", "k_raw", "v_raw", "conv_weight", "cu_seqlens", "conv_init"):
            setattr(c, name, getattr(c, name).cuda())
        return c
    case = on_gpu(workloads.make_prologue([37], H=H, seed=9))
    full = on_gpu(workloads.make_prologue([38], H=H, seed=9))  # same CPU streams: token 37 appended
    assert torch.equal(full.q_raw[:37], case.q_raw)
    _, _, _, fin = _run(case)
    qf, kf, vf, _ = binding.prologue(full.q_raw, full.k_raw, full.v_raw, full.conv_weight, full.cu_seqlens,
                                     full.conv_init, l2_eps=EPS)
    # decode with beta = 0 and no decay leaves the state alone: out = S0^T q~ reveals q~ through S0 = I
    S0 = torch.eye(128, device="cuda").expand(1, H, 128, 128).contiguous()
    la = torch.zeros((1, H, 128), device="cuda")
    beta = torch.zeros((1, H), device="cuda")
    cs = fin.clone()
    out = binding.decode_ex(full.q_raw[37:], full.k_raw[37:], full.v_raw[37:], beta, S0, log_alpha=la,
                            conv_weight=full.conv_weight, conv_state=cs, l2_eps=EPS)
    binding.check_device_error()
    _close(out, qf[37:].double().cpu().numpy(), torch.bfloat16)  # qf went through one bf16 rounding
    assert torch.equal(cs[0, :, 2, :128], full.q_raw[37])


def test_prefill_pass_many_short_sequences():
    """1,500 sequences of 0 to 4 tokens: tiles spanning many sequence starts, and more sequence
    offsets than the kernel keeps in shared memory."""
    lengths = [int(x) for x in np.random.default_rng(12).integers(0, 5, size=1500)]
    case = workloads.make_prologue(lengths, H=2, device="cuda", seed=12)
    _check(case, torch.bfloat16)


@pytest.mark.parametrize("d_k,d_v", [(64, 96), (128, 32)])
def test_decode_step_with_conv_state_odd_sizes(d_k, d_v):
    B, H = 3, 2
    dtype = torch.float32
    st0 = workloads.make_decode_state(B, H, d_k, d_v, device="cuda", seed=13)
    cs0 = workloads.make_conv_state(B, H, d_k, d_v, dtype=dtype, device="cuda", seed=13)
    w = workloads.make_conv_weight(H, d_k, d_v, device="cuda", seed=13)
    step = workloads.make_decode_step(0, B, H, d_k, d_v, dtype=dtype, device="cuda", seed=14)
    state, cs = st0.clone(), cs0.clone()
    out = binding.decode_ex(step.q, step.k, step.v, step.beta, state, log_alpha=step.log_alpha, conv_weight=w,
                            conv_state=cs, l2_eps=EPS)
    binding.check_device_error()
    cu = np.arange(B + 1)
    q, k, v, fin = kda_prologue(cpu(step.q), cpu(step.k), cpu(step.v), cpu(w), cu, cpu(cs0), eps=EPS)
    o_ref, f_ref = kda_recurrent(q, k, v, cpu(step.log_alpha), cpu(step.beta), cu, init_state=cpu(st0))
    assert np.array_equal(cs.double().cpu().numpy(), fin)
    assert rel_max_err(out, o_ref) <= TOL_F32 and rel_max_err(state, f_ref) <= TOL_F32
