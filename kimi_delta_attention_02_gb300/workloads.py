"""Seeded synthetic inputs for KDA prefill and decode.

This module holds input recipes only -- none of the recurrence's arithmetic.
Both the CUDA path (tests, bench, smoke) and the CPU oracle receive exactly the
tensors generated here, so any difference between them comes from the
computation, never from the data.

Recipe (the pages publish no dataset; every workload is synthetic):

* q, k ~ N(0, 1), then L2-normalised over the channel axis for each
  (token, head) in fp32 (Kimi K3 -- Architecture Notes, section 1.1: q and k
  are L2-normalised before the recurrence), then cast to the workload dtype.
* v ~ N(0, 1), cast to the workload dtype.
* log_alpha = -softplus(N(0, 1)) in fp32, per channel, NOT clamped here (the
  kernel applies the lower bound). The "split" mode draws half the heads near
  the -5 bound (-5 + 0.25 N(0,1): about half the values fall below it) and the
  other half near zero (-0.01 softplus(N(0,1))).
* beta = sigmoid(N(0, 1)) in fp32, one per (token, head).
* initial state: zeros, or 0.02 N(0, 1) in fp32 per (sequence, head).
* gated form (decay logits instead of log_alpha): z = -1 + 2 N(0, 1) per
  channel, cast to the workload dtype, and one log-scale A_h = 0.5 N(0, 1) per
  head in fp32. Through g = -5 Sigmoid(e^{A_h} z) this spreads the retention
  over nearly the whole bounded range (alpha from about e^-5 to 1).
* output gate: gate logits r ~ N(0, 1) per value channel, cast to the workload
  dtype (standing in for W_g x), and one RMSNorm weight w = 1 + 0.1 N(0, 1) per
  value channel in fp32 (a weight near its initial value of ones).
* input prologue: raw projections q, k, v ~ N(0, 1) in the workload dtype (not
  normalised: the prologue normalises), convolution weights 0.5 N(0, 1) per
  (head, channel, tap) in fp32, and convolution states (three earlier raw
  inputs) ~ N(0, 1) in the workload dtype.

Every (tensor, head[, step]) pair draws from its own ``torch.Generator``
stream, so any single head can be regenerated without the others and large
workloads are produced one head at a time.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

# tensor ids used to derive stream seeds
_Q, _K, _V, _LA, _BETA, _INIT, _Z, _A, _R, _W, _CW, _CS = 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12


def _stream(seed: int, tensor_id: int, head: int, step: int, device) -> torch.Generator:
    gen = torch.Generator(device=device)
    gen.manual_seed(((seed * 131 + tensor_id) * 1_000_003 + head) * 10_007 + step)
    return gen


def _randn(shape, seed, tensor_id, head, step, device):
    return torch.randn(shape, generator=_stream(seed, tensor_id, head, step, device),
                       device=device, dtype=torch.float32)


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True)


@dataclass
class PrefillCase:
    """One packed varlen prefill problem. Token-major layouts:
    q, k [T_tot, H, d_k]; v [T_tot, H, d_v] (dtype); log_alpha [T_tot, H, d_k] fp32;
    beta [T_tot, H] fp32; cu_seqlens [N+1] int32; init_state [N, H, d_k, d_v] fp32 or None;
    gated form only: z [T_tot, H, d_k] (dtype) and A_log [H] fp32; output gate only:
    out_gate [T_tot, H, d_v] (dtype) and norm_weight [d_v] fp32."""
    name: str
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    log_alpha: torch.Tensor
    beta: torch.Tensor
    cu_seqlens: torch.Tensor
    init_state: torch.Tensor | None
    lengths: list = field(default_factory=list)
    z: torch.Tensor | None = None
    A_log: torch.Tensor | None = None
    out_gate: torch.Tensor | None = None
    norm_weight: torch.Tensor | None = None

    @property
    def total_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def num_seqs(self) -> int:
        return len(self.lengths)


def make_prefill(lengths, H: int, d_k: int = 128, d_v: int = 128, *, dtype=torch.bfloat16,
                 device="cpu", seed: int = 0, init_std: float | None = 0.02,
                 log_alpha_mode: str = "softplus", name: str = "prefill", gated: bool = False,
                 out_gate: bool = False) -> PrefillCase:
    """Generate a packed prefill problem. ``init_std=None`` means no initial state;
    ``gated`` adds the gated form's decay logits z and log-scales A_log; ``out_gate``
    adds the output gate's logits and RMSNorm weight."""
    lengths = [int(x) for x in lengths]
    T = int(sum(lengths))
    N = len(lengths)
    q = torch.empty((T, H, d_k), dtype=dtype, device=device)
    k = torch.empty((T, H, d_k), dtype=dtype, device=device)
    v = torch.empty((T, H, d_v), dtype=dtype, device=device)
    la = torch.empty((T, H, d_k), dtype=torch.float32, device=device)
    beta = torch.empty((T, H), dtype=torch.float32, device=device)
    for h in range(H):
        q[:, h] = _unit_rows(_randn((T, d_k), seed, _Q, h, 0, device)).to(dtype)
        k[:, h] = _unit_rows(_randn((T, d_k), seed, _K, h, 0, device)).to(dtype)
        v[:, h] = _randn((T, d_v), seed, _V, h, 0, device).to(dtype)
        z = _randn((T, d_k), seed, _LA, h, 0, device)
        if log_alpha_mode == "softplus":
            la[:, h] = -torch.nn.functional.softplus(z)
        elif log_alpha_mode == "split":
            la[:, h] = (-5.0 + 0.25 * z) if h < H // 2 else (-0.01 * torch.nn.functional.softplus(z))
        else:
            raise ValueError(f"unknown log_alpha_mode {log_alpha_mode!r}")
        beta[:, h] = torch.sigmoid(_randn((T,), seed, _BETA, h, 0, device))
    init = None
    if init_std is not None:
        init = torch.empty((N, H, d_k, d_v), dtype=torch.float32, device=device)
        for h in range(H):
            init[:, h] = init_std * _randn((N, d_k, d_v), seed, _INIT, h, 0, device)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32), device=device)
    case = PrefillCase(name, q, k, v, la, beta, cu, init, lengths)
    if gated:
        case.z = torch.empty((T, H, d_k), dtype=dtype, device=device)
        case.A_log = torch.empty((H,), dtype=torch.float32, device=device)
        for h in range(H):
            case.z[:, h] = (-1.0 + 2.0 * _randn((T, d_k), seed, _Z, h, 0, device)).to(dtype)
            case.A_log[h] = 0.5 * _randn((1,), seed, _A, h, 0, device)[0]
    if out_gate:
        case.out_gate = torch.empty((T, H, d_v), dtype=dtype, device=device)
        for h in range(H):
            case.out_gate[:, h] = _randn((T, d_v), seed, _R, h, 0, device).to(dtype)
        case.norm_weight = 1.0 + 0.1 * _randn((d_v,), seed, _W, 0, 0, device)
    return case


def varlen_lengths(num_seqs: int = 8, lo: int = 1024, hi: int = 32768, seed: int = 0):
    """Sequence lengths drawn uniformly from [lo, hi] inclusive (numpy PCG64, seeded)."""
    return [int(x) for x in np.random.default_rng(seed).integers(lo, hi + 1, size=num_seqs)]


def sampled_heads(H: int = 32, count: int = 4, seed: int = 0):
    """The seeded head sample checked on the long-context workload."""
    return sorted(int(x) for x in np.random.default_rng(seed).permutation(H)[:count])


# The named prefill workloads: the configurations the tests and the benchmark use (the graded
# shapes plus the gated-decay and output-gate variants of the K3 layer). Each entry: builder kwargs.
PREFILL_WORKLOADS = {
    "prefill_f32_T256_H2": dict(lengths=[256], H=2, dtype=torch.float32, init_std=None),
    "prefill_k3_T4096_H96": dict(lengths=[4096], H=96, dtype=torch.bfloat16, init_std=0.02),
    "prefill_varlen8_H96": dict(lengths=None, H=96, dtype=torch.bfloat16, init_std=0.02,
                                log_alpha_mode="split"),
    "prefill_long_T1M_H32": dict(lengths=[1 << 20], H=32, dtype=torch.bfloat16, init_std=None),
    # the gated decay form on the K3-shaped layer
    "prefill_k3_gated_T4096_H96": dict(lengths=[4096], H=96, dtype=torch.bfloat16, init_std=0.02, gated=True),
    # the K3-shaped layer with the gated decay and the output gate (bf16 output)
    "prefill_k3_outgate_T4096_H96": dict(lengths=[4096], H=96, dtype=torch.bfloat16, init_std=0.02, gated=True,
                                         out_gate=True),
}


def prefill_workload(name: str, device="cpu", seed: int = 0) -> PrefillCase:
    kw = dict(PREFILL_WORKLOADS[name])
    if kw["lengths"] is None:
        kw["lengths"] = varlen_lengths(seed=seed)
    return make_prefill(device=device, seed=seed, name=name, **kw)


@dataclass
class DecodeStep:
    """Inputs of one decode step for B independent sequences: q, k [B, H, d_k],
    v [B, H, d_v] (dtype); log_alpha [B, H, d_k] fp32; beta [B, H] fp32; gated form
    only: z [B, H, d_k] (dtype) and A_log [H] fp32 (a per-head parameter, the same
    for every step)."""
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    log_alpha: torch.Tensor
    beta: torch.Tensor
    z: torch.Tensor | None = None
    A_log: torch.Tensor | None = None
    out_gate: torch.Tensor | None = None
    norm_weight: torch.Tensor | None = None


def make_decode_state(B: int, H: int, d_k: int = 128, d_v: int = 128, *, device="cpu", seed: int = 0,
                      init_std: float = 0.02) -> torch.Tensor:
    state = torch.empty((B, H, d_k, d_v), dtype=torch.float32, device=device)
    for h in range(H):
        state[:, h] = init_std * _randn((B, d_k, d_v), seed, _INIT, h, 0, device)
    return state


def make_decode_step(step: int, B: int, H: int, d_k: int = 128, d_v: int = 128, *,
                     dtype=torch.bfloat16, device="cpu", seed: int = 0, gated: bool = False,
                     out_gate: bool = False) -> DecodeStep:
    """Fresh inputs for decode step ``step`` (streams differ per step)."""
    s = step + 1
    q = _unit_rows(_randn((B, H, d_k), seed, _Q, 0, s, device)).to(dtype)
    k = _unit_rows(_randn((B, H, d_k), seed, _K, 0, s, device)).to(dtype)
    v = _randn((B, H, d_v), seed, _V, 0, s, device).to(dtype)
    la = -torch.nn.functional.softplus(_randn((B, H, d_k), seed, _LA, 0, s, device))
    beta = torch.sigmoid(_randn((B, H), seed, _BETA, 0, s, device))
    st = DecodeStep(q, k, v, la, beta)
    if gated:
        st.z = (-1.0 + 2.0 * _randn((B, H, d_k), seed, _Z, 0, s, device)).to(dtype)
        st.A_log = 0.5 * _randn((H,), seed, _A, 0, 0, device)
    if out_gate:
        st.out_gate = _randn((B, H, d_v), seed, _R, 0, s, device).to(dtype)
        st.norm_weight = 1.0 + 0.1 * _randn((d_v,), seed, _W, 0, 0, device)
    return st


DECODE_WORKLOAD = dict(B=256, H=96, d_k=128, d_v=128, steps=64, dtype=torch.bfloat16)


@dataclass
class PrologueCase:
    """Raw projections for the input prologue over packed sequences: q_raw, k_raw [T_tot, H, d_k],
    v_raw [T_tot, H, d_v] (dtype); conv_weight [H, 2 d_k + d_v, 4] fp32; cu_seqlens [N+1] int32;
    conv_init [N, H, 3, 2 d_k + d_v] (dtype) or None."""
    q_raw: torch.Tensor
    k_raw: torch.Tensor
    v_raw: torch.Tensor
    conv_weight: torch.Tensor
    cu_seqlens: torch.Tensor
    conv_init: torch.Tensor | None
    lengths: list = field(default_factory=list)


def make_conv_weight(H: int, d_k: int = 128, d_v: int = 128, *, device="cpu", seed: int = 0) -> torch.Tensor:
    C3 = 2 * d_k + d_v
    w = torch.empty((H, C3, 4), dtype=torch.float32, device=device)
    for h in range(H):
        w[h] = 0.5 * _randn((C3, 4), seed, _CW, h, 0, device)
    return w


def make_conv_state(N: int, H: int, d_k: int = 128, d_v: int = 128, *, dtype=torch.bfloat16, device="cpu",
                    seed: int = 0) -> torch.Tensor:
    st = torch.empty((N, H, 3, 2 * d_k + d_v), dtype=dtype, device=device)
    for h in range(H):
        st[:, h] = _randn((N, 3, 2 * d_k + d_v), seed, _CS, h, 0, device).to(dtype)
    return st


def make_prologue(lengths, H: int, d_k: int = 128, d_v: int = 128, *, dtype=torch.bfloat16, device="cpu",
                  seed: int = 0, with_state: bool = True) -> PrologueCase:
    lengths = [int(x) for x in lengths]
    T = int(sum(lengths))
    q = torch.empty((T, H, d_k), dtype=dtype, device=device)
    k = torch.empty((T, H, d_k), dtype=dtype, device=device)
    v = torch.empty((T, H, d_v), dtype=dtype, device=device)
    for h in range(H):
        q[:, h] = _randn((T, d_k), seed, _Q, h, 0, device).to(dtype)
        k[:, h] = _randn((T, d_k), seed, _K, h, 0, device).to(dtype)
        v[:, h] = _randn((T, d_v), seed, _V, h, 0, device).to(dtype)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32), device=device)
    st = make_conv_state(len(lengths), H, d_k, d_v, dtype=dtype, device=device, seed=seed) if with_state else None
    return PrologueCase(q, k, v, make_conv_weight(H, d_k, d_v, device=device, seed=seed), cu, st, lengths)
