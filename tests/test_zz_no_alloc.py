"""kda_prefill_noalloc: the prefill for callers that cannot allocate device memory (a serving
engine that owns the whole GPU in its own pool, a plugin inside a framework that owns every
allocation, a latency-critical region where cudaMalloc would stall the device). Its scratch is an
array inside the library, shared by every call. The GPU test calls it through the C ABI twice in
a row, on different inputs, and compares each result with kda_prefill given a workspace; the CPU
test checks that sizes beyond the array are refused before anything is enqueued. This file sorts
last so that a run stopping at its first failure has run every other test already."""

import ctypes

import pytest
import torch

from helpers import TOL_BF16, rel_max_err
from kimi_delta_attention_02_gb300 import binding as B
from kimi_delta_attention_02_gb300 import workloads

SCRATCH_BYTES = 16 << 20


@pytest.mark.gpu
@pytest.mark.parametrize("lengths,H", [([20000], 32), ([40, 3000, 0, 777, 2048, 129] * 4, 8)])
def test_noalloc_matches_prefill_on_two_calls_in_a_row(lengths, H):
    """One sequence in 3 segments (12 MiB of scratch, the same as T = 2^20 with H = 32), and 24
    packed sequences taken longest first; each call's inputs differ from the previous call's, so
    scratch left over from it would show."""
    T = sum(lengths)
    assert 0 < B.workspace_size(T, len(lengths), H) <= SCRATCH_BYTES
    for seed in (70, 71):
        case = workloads.make_prefill(lengths, H=H, device="cuda", seed=seed)
        args = (case.q, case.k, case.v, case.log_alpha, case.beta, case.cu_seqlens, case.init_state)
        ref, ref_fin = B.prefill(*args, workspace="auto")
        out = torch.full_like(ref, float("nan"))
        fin = torch.full_like(ref_fin, float("nan"))
        B.prefill_noalloc(*args, out=out, final_state=fin)
        B.check_device_error()
        assert rel_max_err(out, ref.double().cpu().numpy()) <= TOL_BF16
        assert rel_max_err(fin, ref_fin.double().cpu().numpy()) <= TOL_BF16


def test_noalloc_refuses_sizes_beyond_its_scratch():
    """Host-side fake addresses: the size check runs before any CUDA call. T = 2^20 with 50 heads
    plans 3 segments (19.7 MB), with 76 heads 2 segments (19.9 MB): both above 16 MiB."""
    lib = B.lib()
    a = [(i + 1) << 40 for i in range(8)]  # fake device addresses 1 TiB apart: no two ranges overlap
    for H in (50, 76):
        assert B.workspace_size(1 << 20, 1, H) > SCRATCH_BYTES
        st = lib.kda_prefill_noalloc(a[0], a[1], a[2], a[3], a[4], a[5], 1, 1 << 20, H, 128, 128, B.KDA_BF16,
                                     B.KDA_F32, -5.0, 1.0, None, a[6], a[7], None)
        assert st == B.KDA_ERR_UNSUPPORTED
    # an argument error is reported before the size check
    st = lib.kda_prefill_noalloc(None, a[1], a[2], a[3], a[4], a[5], 1, 1 << 20, 50, 128, 128, B.KDA_BF16,
                                 B.KDA_F32, -5.0, 1.0, None, a[6], a[7], None)
    assert st == B.KDA_ERR_INVALID_ARG
