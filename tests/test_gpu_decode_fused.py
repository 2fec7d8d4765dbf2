"""The fused decode step at the benchmark's size, in the launch `bench.py` times: B=256 sequences,
H=96, bf16 raw q, k, v through the prologue (4-tap convolution over the sequence's state, which is
shifted in place, Swish, L2 norm of q and k; Kimi K3 -- Architecture Notes, section 1.1), the
gated decay (section 1.2), the delta-rule update of the fp32 state and the output gate with
head-wise RMSNorm (section 1.3), bf16 out. Three steps in a row; 48 seeded (sequence, head) pairs
are replayed by the fp64 oracle stage by stage."""

import numpy as np
import pytest
import torch

from helpers import TOL_BF16, cpu, gated_output_err, rel_max_err
from kimi_delta_attention_02_gb300 import binding, workloads
from oracle import kda_prologue, kda_recurrent_gated, output_gate_rmsnorm

pytestmark = pytest.mark.gpu

B, H, STEPS, EPS = 256, 96, 3, 1e-6


def test_fused_decode_benchmark_size():
    state = workloads.make_decode_state(B, H, device="cuda", seed=0)
    conv_w = workloads.make_conv_weight(H, device="cuda", seed=0)
    conv_state = workloads.make_conv_state(B, H, device="cuda", seed=0)
    rng = np.random.default_rng(21)
    pairs = [(int(b), int(h)) for b, h in zip(rng.integers(0, B, 48), rng.integers(0, H, 48))]
    ref_state = {p: cpu(state[p]).double().numpy()[None, None] for p in pairs}  # [1, 1, d_k, d_v]
    ref_conv = {p: cpu(conv_state[p]).double().numpy()[None, None] for p in pairs}  # [1, 1, 3, C3]
    w_cpu = cpu(conv_w)
    cu = np.array([0, 1])
    for s in range(STEPS):
        st = workloads.make_decode_step(s, B, H, dtype=torch.bfloat16, device="cuda", seed=0, gated=True,
                                        out_gate=True)
        out = torch.empty((B, H, 128), dtype=torch.bfloat16, device="cuda")
        binding.decode_ex(st.q, st.k, st.v, st.beta, state, z=st.z, A_log=st.A_log, out_gate=st.out_gate,
                          norm_weight=st.norm_weight, conv_weight=conv_w, conv_state=conv_state, out=out,
                          norm_eps=EPS, l2_eps=EPS)
        binding.check_device_error()
        ys, y_refs, o_refs = [], [], []
        for (b, h) in pairs:
            one = lambda t: cpu(t[b, h]).reshape(1, 1, -1)
            q, k, v, fin = kda_prologue(one(st.q), one(st.k), one(st.v), w_cpu[h:h + 1], cu, ref_conv[(b, h)],
                                        eps=EPS)
            ref_conv[(b, h)] = fin
            o, f = kda_recurrent_gated(q, k, v, one(st.z), cpu(st.A_log)[h:h + 1], cpu(st.beta[b, h]).reshape(1, 1),
                                       cu, init_state=ref_state[(b, h)], num_threads=1)
            ref_state[(b, h)] = f
            y_refs.append(output_gate_rmsnorm(o, one(st.out_gate), cpu(st.norm_weight), EPS))
            o_refs.append(o)
            ys.append(cpu(out[b, h]).double().numpy().reshape(1, 1, -1))
        y, y_ref, o_ref = (np.concatenate(a) for a in (ys, y_refs, o_refs))
        e_y = gated_output_err(y, y_ref, o_ref, bf16_out=True)
        assert e_y <= TOL_BF16, (s, e_y)
    g_state = np.concatenate([cpu(state[p]).double().numpy()[None, None] for p in pairs])
    r_state = np.concatenate([ref_state[p] for p in pairs])
    assert rel_max_err(g_state, r_state) <= TOL_BF16
    for p in pairs:  # the convolution state holds exact copies of the last three raw inputs
        assert np.array_equal(cpu(conv_state[p]).double().numpy(), ref_conv[p][0, 0])
