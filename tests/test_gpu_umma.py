"""tcgen05 MMA descriptor encodings used by the chunked prefill kernel, checked
on the GPU against host matrix products (kda_selftest_umma).

Settings pinned here: 128-byte-swizzled K-major operands (leading byte offset
16, stride byte offset 1024 = one 8-row swizzle atom) for bf16, fp16 and tf32;
MN-major 16-bit operands with leading byte offset = the 64-element block
stride (rows x 128 bytes) and stride byte offset 1024; 64-byte-swizzled K-major
16-bit operands; the negate-A bit; and,
for M = 64, accumulator row m in tensor-memory lane (m mod 16) + 32 (m div 16).
The shapes are the ones the chunk-32 kernel issues."""

import pytest
import torch

from kimi_delta_attention_02_gb300 import binding as B

pytestmark = pytest.mark.gpu


def _round(x, fmt):
    if fmt == "bf16":
        return x.bfloat16().float()
    if fmt == "f16":
        return x.half().float()
    bits = x.float().contiguous().view(torch.int32)  # tf32, round to nearest (ties away from zero)
    bits = (bits + (1 << 12)) & ~((1 << 13) - 1)
    return bits.view(torch.float32)


def _lanes_m64():
    return torch.tensor([(m % 16) + 32 * (m // 16) for m in range(64)])


CASES = [
    # fmt,  M,   N,   K, a_mn, b_mn, neg    use in the chunked kernel (sw64 cases: see SW64_CASES)
    ("tf32", 64, 48, 128, False, False, False),
    ("f16", 128, 32, 32, True, False, False),    # W^T = Kg^T T'^T, Kg token-major
    ("f16", 128, 64, 32, True, False, False),    # [U~^T | 0] = V^T [T'; 0]^T, V token-major
    ("f16", 128, 64, 128, False, True, False),   # [U^T | O^T] += S^T [-W^T | Q~^T] (128-row MN-major B)
    ("f16", 128, 160, 32, False, False, False),  # [O^T | S^T] += U^T [P ; K^^T]^T
    ("tf32", 64, 32, 128, False, False, False),  # Gram: [Q f ; K f] (K g)^T, one reference per chunk
    ("f16", 64, 128, 32, False, True, False),
    ("f16", 128, 32, 128, False, False, True),   # negate-A bit
    ("f16", 128, 128, 32, False, True, False),
    ("bf16", 128, 64, 128, False, False, False),
    ("bf16", 128, 128, 64, False, True, False),
    ("bf16", 64, 32, 128, False, False, False),
]


# 64-byte-swizzled K-major operands (rows of 32 fp16): the half-width tiles of the pipelined kernel
SW64_CASES = [
    ("f16", 128, 32, 32, True, False, False),    # W^T = Kg^T T'^T with T' 64-byte swizzled
    ("f16", 128, 64, 32, True, False, False),    # [U~^T | 0] = V^T [T'; 0]^T
    ("f16", 128, 32, 32, False, False, False),   # O^T += U^T P^T (U^T, P both 64-byte swizzled)
    ("f16", 128, 128, 32, False, False, False),  # S^T += U^T K^ (K^^T rows 64-byte swizzled)
    ("f16", 128, 128, 64, False, False, False),  # two 32-wide K blocks
    ("f16", 128, 160, 32, False, False, False),  # [O^T | S^T] += U^T [P ; K^^T]^T in one product
    ("bf16", 64, 32, 32, False, False, False),
]


@pytest.mark.parametrize("fmt,M,N,K,a_mn,b_mn,neg", SW64_CASES)
def test_umma_layouts_sw64(fmt, M, N, K, a_mn, b_mn, neg):
    _check(fmt, M, N, K, a_mn, b_mn, neg, sw64=True)


@pytest.mark.parametrize("fmt,M,N,K,a_mn,b_mn,neg", CASES)
def test_umma_layouts(fmt, M, N, K, a_mn, b_mn, neg):
    _check(fmt, M, N, K, a_mn, b_mn, neg, sw64=False)


def _check(fmt, M, N, K, a_mn, b_mn, neg, sw64):
    g = torch.Generator(device="cpu").manual_seed(M * 7 + N * 3 + K + 11 * a_mn + 5 * b_mn)
    A = torch.randn(M, K, generator=g)
    Bm = torch.randn(N, K, generator=g)
    E = _round(A, fmt).double() @ _round(Bm, fmt).double().T
    sbo = 512 if sw64 else 1024  # one 8-row swizzle atom
    kw = dict(fmt=fmt, sw64=sw64, a_mn_major=a_mn, b_mn_major=b_mn, negate_a=neg, a_lbo=16,
              a_sbo=1024 if a_mn else sbo, b_lbo=16, b_sbo=1024 if b_mn else sbo)
    if a_mn:
        kw["a_lbo"] = K * 128  # block of 64 M-elements holds K rows of 128 bytes
    if b_mn:
        kw["b_lbo"] = K * 128
    D = B.selftest_umma(A.cuda(), Bm.cuda(), M, N, K, **kw).cpu().double()
    got = D if M == 128 else D[_lanes_m64()]
    want = -E if neg else E
    assert (got - want).abs().max().item() < 1e-4 * max(1.0, want.abs().max().item())
    B.check_device_error()
