"""The seeded generators: determinism, per-head streams and the input recipe."""

import torch

from kimi_delta_attention_02_gb300 import workloads as W


def test_deterministic_and_seed_sensitive():
    a = W.make_prefill([37, 5], H=3, d_k=16, d_v=8, seed=0)
    b = W.make_prefill([37, 5], H=3, d_k=16, d_v=8, seed=0)
    c = W.make_prefill([37, 5], H=3, d_k=16, d_v=8, seed=1)
    for name in ("q", "k", "v", "log_alpha", "beta", "init_state"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
        assert not torch.equal(getattr(a, name), getattr(c, name)), name


def test_heads_are_independent_streams():
    """Head h's data does not depend on how many heads are generated."""
    a = W.make_prefill([20], H=2, d_k=8, d_v=8, dtype=torch.float32)
    b = W.make_prefill([20], H=5, d_k=8, d_v=8, dtype=torch.float32)
    for name in ("q", "k", "v", "log_alpha", "beta"):
        assert torch.equal(getattr(a, name), getattr(b, name)[:, :2]), name
    assert torch.equal(a.init_state, b.init_state[:, :2])


def test_recipe_properties():
    case = W.make_prefill([300], H=4, d_k=32, d_v=16, dtype=torch.bfloat16)
    qn = case.q.float().norm(dim=-1)
    assert torch.all((qn - 1).abs() < 1e-2)
    assert torch.all(case.log_alpha < 0)
    assert torch.all((case.beta > 0) & (case.beta < 1))
    assert case.cu_seqlens.dtype == torch.int32 and case.cu_seqlens.tolist() == [0, 300]
    split = W.make_prefill([400], H=4, d_k=32, d_v=16, log_alpha_mode="split")
    strong, weak = split.log_alpha[:, :2], split.log_alpha[:, 2:]
    assert abs(strong.mean().item() + 5.0) < 0.05 and 0.3 < (strong < -5).float().mean().item() < 0.7
    assert torch.all(weak < 0) and torch.all(weak > -0.2)


def test_varlen_lengths_and_head_sample():
    lengths = W.varlen_lengths()
    assert len(lengths) == 8 and all(1024 <= L <= 32768 for L in lengths)
    assert lengths == W.varlen_lengths()
    heads = W.sampled_heads()
    assert len(heads) == 4 and len(set(heads)) == 4 and all(0 <= h < 32 for h in heads)


def test_decode_steps_differ():
    s0 = W.make_decode_step(0, 4, 2, 8, 8)
    s1 = W.make_decode_step(1, 4, 2, 8, 8)
    assert not torch.equal(s0.q, s1.q)
    st = W.make_decode_state(4, 2, 8, 8)
    assert st.shape == (4, 2, 8, 8) and abs(st.std().item() - 0.02) < 0.005
