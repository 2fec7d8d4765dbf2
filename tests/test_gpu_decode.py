"""kda_decode on the GPU against the fp64 oracle.

A decode step is the recurrence over B one-token sequences, so B decode steps
chained on one (sequence, head) are a prefill of that many tokens: the oracle
replays each sampled pair's steps as one sequence."""

import numpy as np
import pytest
import torch

from helpers import rel_max_err, tol_for
from kimi_delta_attention_02_gb300 import binding, workloads
from oracle import kda_recurrent

pytestmark = pytest.mark.gpu


def _run_and_check(B, H, d_k, d_v, steps, dtype, pairs=None, seed=0):
    dev = torch.device("cuda")
    state0 = workloads.make_decode_state(B, H, d_k, d_v, device=dev, seed=seed)
    state = state0.clone()
    if pairs is None:
        pairs = [(b, h) for b in range(B) for h in range(H)]
    bi = torch.tensor([p[0] for p in pairs], device=dev)
    hi = torch.tensor([p[1] for p in pairs], device=dev)
    seq = {name: [] for name in ("q", "k", "v", "log_alpha", "beta", "out")}
    for s in range(steps):
        st = workloads.make_decode_step(s, B, H, d_k, d_v, dtype=dtype, device=dev, seed=seed)
        out = binding.decode(st.q, st.k, st.v, st.log_alpha, st.beta, state)
        for name in ("q", "k", "v", "log_alpha", "beta"):
            seq[name].append(getattr(st, name)[bi, hi].cpu())
        seq["out"].append(out[bi, hi].cpu())
    binding.check_device_error()
    P = len(pairs)
    # sequence p = the sampled pair's steps in order: token-major [P*steps, 1, d]
    stack = lambda xs: torch.stack(xs, dim=1).reshape(P * steps, 1, -1)
    cu = np.arange(0, P * steps + 1, steps, dtype=np.int64)
    beta = torch.stack(seq["beta"], dim=1).reshape(P * steps, 1)
    init = state0[bi, hi].cpu().reshape(P, 1, d_k, d_v)
    o_ref, f_ref = kda_recurrent(stack(seq["q"]), stack(seq["k"]), stack(seq["v"]), stack(seq["log_alpha"]), beta,
                                 cu, init_state=init)
    o_gpu = stack(seq["out"])
    f_gpu = state[bi, hi].cpu().reshape(P, 1, d_k, d_v)
    tol = tol_for(dtype)
    e_o, e_f = rel_max_err(o_gpu, o_ref), rel_max_err(f_gpu, f_ref)
    assert e_o <= tol and e_f <= tol, (e_o, e_f)
    return e_o, e_f


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_small_all_pairs(dtype):
    _run_and_check(B=6, H=3, d_k=128, d_v=128, steps=5, dtype=dtype)


@pytest.mark.parametrize("d_k,d_v", [(64, 32), (128, 64), (16, 128), (100, 4)])
def test_decode_odd_head_dims(d_k, d_v):
    _run_and_check(B=3, H=2, d_k=d_k, d_v=d_v, steps=3, dtype=torch.float32)


def test_decode_full_workload_sampled_pairs():
    """B=256 sequences, H=96, d=128, bf16, 64 in-place steps; 64 seeded pairs checked."""
    cfg = workloads.DECODE_WORKLOAD
    rng = np.random.default_rng(0)
    pairs = sorted({(int(b), int(h)) for b, h in zip(rng.integers(0, cfg["B"], 64), rng.integers(0, cfg["H"], 64))})
    _run_and_check(cfg["B"], cfg["H"], cfg["d_k"], cfg["d_v"], cfg["steps"], cfg["dtype"], pairs=pairs)


def test_decode_matches_recurrent_prefill():
    """N decode steps on one sequence equal a prefill of those N tokens (GPU vs GPU, tight)."""
    dev = torch.device("cuda")
    B, H, steps = 1, 4, 7
    st0 = workloads.make_decode_state(B, H, device=dev)
    state = st0.clone()
    qs, ks, vs, las, bs, outs = [], [], [], [], [], []
    for s in range(steps):
        st = workloads.make_decode_step(s, B, H, dtype=torch.float32, device=dev)
        outs.append(binding.decode(st.q, st.k, st.v, st.log_alpha, st.beta, state))
        qs.append(st.q[0]); ks.append(st.k[0]); vs.append(st.v[0]); las.append(st.log_alpha[0]); bs.append(st.beta[0])
    cu = torch.tensor([0, steps], dtype=torch.int32, device=dev)
    o, f = binding.prefill(torch.stack(qs), torch.stack(ks), torch.stack(vs), torch.stack(las), torch.stack(bs),
                           cu, st0, recurrent=True)
    assert rel_max_err(torch.stack(outs)[:, 0], o.double().cpu().numpy()) < 1e-5
    assert rel_max_err(state, f.double().cpu().numpy()) < 1e-5
