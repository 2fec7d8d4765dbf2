"""tcgen05 MMA descriptor encodings used by the chunked prefill kernel, checked
on the GPU against host matrix products (kda_selftest_umma).

Settings pinned here: 128-byte-swizzled K-major operands (leading byte offset
16, stride byte offset 1024 = one 8-row swizzle atom); MN-major operands with
leading byte offset = the 64-element block stride and stride byte offset 1024;
the negate-A bit; and, for M = 64, accumulator row m in tensor-memory lane
(m mod 16) + 32 * (m div 16)."""

import pytest
import torch

from kimi_delta_attention_02_gb300 import binding as B

pytestmark = pytest.mark.gpu


def _mats(M, N, K, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    A = torch.randn(M, K, generator=g).bfloat16()
    Bm = torch.randn(N, K, generator=g).bfloat16()
    return A, Bm, A.float() @ Bm.float().T


def _lanes_m64():
    return torch.tensor([(m % 16) + 32 * (m // 16) for m in range(64)])


@pytest.mark.parametrize("M,N,K,a_mn,b_mn,neg", [
    (128, 64, 128, False, False, False),   # S^T W^T and S^T Q~^T
    (128, 64, 128, False, False, True),    # U~^T - S^T W^T (negated A)
    (128, 64, 64, False, False, False),    # U^T P^T
    (128, 128, 64, False, True, False),    # U^T K^ (K^ token-major)
    (128, 64, 64, True, False, False),     # V^T T'^T (V token-major)
    (128, 256, 128, False, False, False),
    (64, 32, 128, False, False, False),    # intra-chunk Gram tiles
    (64, 128, 64, False, True, False),     # W = T' Kg (Kg token-major)
])
def test_umma_layouts(M, N, K, a_mn, b_mn, neg):
    A, Bm, E = _mats(M, N, K, seed=M + N + K + 7 * a_mn + 3 * b_mn)
    kw = dict(a_mn_major=a_mn, b_mn_major=b_mn, negate_a=neg, a_lbo=16, a_sbo=1024, b_lbo=16, b_sbo=1024)
    if a_mn:
        kw["a_lbo"] = K * 128  # block of 64 M-elements holds K rows of 128 bytes
    if b_mn:
        kw["b_lbo"] = K * 128
    D = B.selftest_umma(A.cuda(), Bm.cuda(), M, N, K, **kw).cpu()
    got = D if M == 128 else D[_lanes_m64()]
    want = -E if neg else E
    assert (got - want).abs().max().item() < 1e-3 * max(1.0, want.abs().max().item())
    B.check_device_error()
