"""The C-ABI library: it loads, exports every declared entry point, and its
host-side argument validation rejects bad calls before touching a GPU."""

import ctypes
import os
import re

import pytest

import __graft_entry__
from kimi_delta_attention_02_gb300 import binding as B

NULL = None


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(B.LIB_PATH):
        __graft_entry__.build()
    return B.lib()


def declared_functions():
    names = []
    for path in B.HEADERS:
        with open(path) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(kda_[a-z_0-9]+)\s*\(", text)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"kda_prefill", "kda_decode", "kda_prefill_recurrent", "kda_check_device_error",
            "kda_status_string", "kda_version", "kda_selftest_umma", "kda_prefill_gated",
            "kda_prefill_gated_recurrent", "kda_decode_gated", "kda_prefill_ex", "kda_decode_ex",
            "kda_prologue", "kda_selftest_wait_timeout", "kda_prefill_workspace_size"} <= set(names)
    for name in names:
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    assert B.status_string(0) == "KDA_OK"
    assert B.status_string(4) == "KDA_ERR_TIMEOUT"
    assert B.status_string(5) == "KDA_ERR_RANGE"
    assert B.status_string(99) == "KDA_ERR_UNKNOWN"
    assert lib.kda_version() >= 100


def _prefill(lib, fn="kda_prefill", **over):
    """Call with host-side fake addresses: validation must reject before any CUDA call."""
    a = dict(q=0x10000, k=0x20000, v=0x30000, la=0x40000, beta=0x50000, cu=0x60000, N=1, T=4, H=2, dk=128,
             dv=128, dtype=1, odtype=0, lb=-5.0, scale=1.0, init=NULL, out=0x70000, fin=0x80000, ws=NULL,
             ws_bytes=0, stream=NULL)
    a.update(over)
    args = [a["q"], a["k"], a["v"], a["la"], a["beta"], a["cu"], a["N"], a["T"], a["H"], a["dk"], a["dv"], a["dtype"],
            a["odtype"], a["lb"], a["scale"], a["init"], a["out"], a["fin"]]
    if fn == "kda_prefill":
        args += [a["ws"], a["ws_bytes"]]
    return getattr(lib, fn)(*args, a["stream"])


@pytest.mark.parametrize("fn", ["kda_prefill", "kda_prefill_recurrent"])
@pytest.mark.parametrize("over,expect", [
    (dict(q=NULL), B.KDA_ERR_INVALID_ARG),
    (dict(cu=NULL), B.KDA_ERR_INVALID_ARG),
    (dict(out=NULL), B.KDA_ERR_INVALID_ARG),
    (dict(q=0x10008), B.KDA_ERR_INVALID_ARG),          # misaligned
    (dict(cu=0x60002), B.KDA_ERR_INVALID_ARG),
    (dict(dtype=7), B.KDA_ERR_INVALID_ARG),
    (dict(odtype=3), B.KDA_ERR_INVALID_ARG),
    (dict(H=0), B.KDA_ERR_INVALID_ARG),
    (dict(N=-1), B.KDA_ERR_INVALID_ARG),
    (dict(T=-1), B.KDA_ERR_INVALID_ARG),
    (dict(dk=129), B.KDA_ERR_UNSUPPORTED),
    (dict(dv=0), B.KDA_ERR_INVALID_ARG),
    (dict(T=1 << 31), B.KDA_ERR_UNSUPPORTED),
    (dict(out=0x10000), B.KDA_ERR_INVALID_ARG),       # output aliases an input
    (dict(fin=0x40000), B.KDA_ERR_INVALID_ARG),
    (dict(init=0x90000, fin=0x90000 + 4096), B.KDA_ERR_INVALID_ARG),  # partial overlap
])
def test_prefill_rejects(lib, fn, over, expect):
    assert _prefill(lib, fn, **over) == expect


@pytest.mark.parametrize("over", [
    dict(ws=0x1000000, ws_bytes=0),                 # a workspace pointer without bytes
    dict(ws=NULL, ws_bytes=4096),                   # bytes without a pointer
    dict(ws=0x1000008, ws_bytes=4096),              # misaligned
    dict(ws=0x70000, ws_bytes=4096),                # over the output
    dict(ws=0x60000 - 16, ws_bytes=32),             # over cu_seqlens
    dict(ws=0x80000 + 65536, ws_bytes=16),          # inside the final state
])
def test_prefill_rejects_bad_workspace(lib, over):
    assert _prefill(lib, **over) == B.KDA_ERR_INVALID_ARG


def test_workspace_size_is_a_pure_host_query(lib):
    # no CUDA call: it answers on a machine without a GPU, the same way every time
    for args in [(4096, 1, 96, 128, 128), (1 << 20, 1, 32, 128, 128), (135000, 8, 96, 128, 128), (0, 0, 1, 1, 1)]:
        a = lib.kda_prefill_workspace_size(*args)
        assert a == lib.kda_prefill_workspace_size(*args)
        assert a % 16 == 0


def _planned_workspace(T, N, H, d_k=128, d_v=128):
    """The schedules' workspace, restated from their plan: one sequence is cut into the largest
    number m >= 2 of segments whose passes (pass 1: 2m - 3 runs, or 1 for m = 2; pass 3: m runs)
    each fit one CTA per SM on 152 SMs, with segments (whole 32-token chunks) of at least 4096
    tokens and at most 64 runs; its maps take max(runs, m) + m states of 128 x 128 fp32 per
    head, each part rounded up to 256 bytes. Several sequences take the longest-first order
    (4 bytes each, rounded up to 256) once their chains outnumber the SMs (at most 8192)."""
    up256 = lambda n: (n + 255) // 256 * 256
    state = 128 * 128 * 4
    if d_k != 128 or d_v != 128 or H < 1 or T <= 0:
        return 0
    if N == 1:
        best = None
        for m in range(2, 65):
            runs = 1 if m == 2 else 2 * m - 3
            if runs > 64 or H * runs > 152 or H * m > 152:
                break
            L = ((T + m - 1) // m + 31) // 32 * 32
            if L < 4096 or (m - 1) * L >= T:
                break
            best = (m, runs)
        if best is None:
            return 0
        m, runs = best
        return up256(max(runs, m) * H * state) + up256(m * H * state)
    return up256(4 * N) if 1 < N <= 8192 and N * H > 152 else 0


@pytest.mark.parametrize("T,N,H", [(1 << 20, 1, 32), (1 << 20, 1, 1), (1 << 20, 1, 96), (1 << 16, 1, 32),
                                   (8192, 1, 8), (8191, 1, 8), (4096, 1, 96), (135000, 8, 96), (10000, 2, 76),
                                   (10000, 2, 77), (10000, 200, 1), (10000, 9000, 1)])
def test_workspace_sizes_follow_the_schedule_plan(lib, T, N, H):
    assert lib.kda_prefill_workspace_size(T, N, H, 128, 128) == _planned_workspace(T, N, H)


def test_workspace_of_the_long_context_shape(lib):
    # T = 2^20, H = 32: three segments (pass 1 runs 3 chains per head; four segments would need
    # 5 x 32 = 160 > 152 CTAs in pass 1), so 3 + 3 states per head: 6 x 32 x 64 KiB = 12 MiB
    assert lib.kda_prefill_workspace_size(1 << 20, 1, 32, 128, 128) == 6 * 32 * 65536
    assert lib.kda_prefill_workspace_size(1 << 20, 1, 32, 64, 128) == 0


def test_prefill_accepts_empty_work(lib):
    # zero sequences and zero tokens: nothing to enqueue, no CUDA call is made
    assert _prefill(lib, N=0, T=0, q=NULL, k=NULL, v=NULL, la=NULL, beta=NULL, out=NULL, fin=NULL) == B.KDA_OK


@pytest.mark.parametrize("over,expect", [
    (dict(state=NULL), B.KDA_ERR_INVALID_ARG),
    (dict(B=0), B.KDA_ERR_INVALID_ARG),
    (dict(dv=6), B.KDA_ERR_UNSUPPORTED),
    (dict(dk=256), B.KDA_ERR_UNSUPPORTED),
    (dict(state=0x1000004), B.KDA_ERR_INVALID_ARG),
    (dict(dtype=2), B.KDA_ERR_INVALID_ARG),
    (dict(odtype=-1), B.KDA_ERR_INVALID_ARG),
    (dict(state=0x10000), B.KDA_ERR_INVALID_ARG),        # the state over q
    (dict(state=0x40000 - 4096), B.KDA_ERR_INVALID_ARG), # the state running into log_alpha
    (dict(out=0x20000), B.KDA_ERR_INVALID_ARG),          # out over k
    (dict(out=0x50000), B.KDA_ERR_INVALID_ARG),          # out over beta
    (dict(out=0x1000000 + 8192), B.KDA_ERR_INVALID_ARG), # out inside the state
])
def test_decode_rejects(lib, over, expect):
    a = dict(q=0x10000, k=0x20000, v=0x30000, la=0x40000, beta=0x50000, state=0x1000000, out=0x70000, B=2, H=2,
             dk=128, dv=128, dtype=1, odtype=0)
    a.update(over)
    st = lib.kda_decode(a["q"], a["k"], a["v"], a["la"], a["beta"], a["state"], a["out"], a["B"], a["H"], a["dk"],
                        a["dv"], a["dtype"], a["odtype"], -5.0, 1.0, NULL)
    assert st == expect


def test_selftest_rejects_bad_shapes(lib):
    st = lib.kda_selftest_umma(0x1000, 0x2000, 0x3000, 96, 64, 64, 1, 0, 0, 0, 0, 16, 1024, 16, 1024, 0x4000, NULL)
    assert st == B.KDA_ERR_UNSUPPORTED
    st = lib.kda_selftest_umma(0x1000, 0x2000, 0x3000, 128, 64, 64, 2, 0, 1, 0, 0, 16, 1024, 16, 1024, 0x4000, NULL)
    assert st == B.KDA_ERR_UNSUPPORTED  # tf32 operands are K-major only
    st = lib.kda_selftest_umma(0x1000, 0x2000, 0x3000, 128, 64, 64, 5, 0, 0, 0, 0, 16, 1024, 16, 1024, 0x4000, NULL)
    assert st == B.KDA_ERR_INVALID_ARG


@pytest.mark.parametrize("args", [
    (128, 64, 64, 1, 0, 0, 0, 0, 16, 32768, 16, 1024),     # K-major A, 16 atoms 32 KB apart: far past its tile
    (128, 64, 128, 1, 0, 0, 0, 0, 16, 1024, 16, 8192),     # K-major B rows 8 KB apart
    (128, 128, 128, 0, 0, 1, 0, 0, 32768, 32768, 16, 1024),  # MN-major A: blocks and K groups 32 KB apart
    (128, 256, 128, 1, 0, 0, 1, 0, 16, 1024, 32768, 1024), # MN-major B, 4 blocks of 64 columns 32 KB apart
])
def test_selftest_rejects_descriptors_outside_the_tile(lib, args):
    M, N, K, fmt, sw64, amn, bmn, neg, albo, asbo, blbo, bsbo = args
    st = lib.kda_selftest_umma(0x1000, 0x2000, 0x3000, M, N, K, fmt, sw64, amn, bmn, neg, albo, asbo, blbo, bsbo,
                               0x4000, NULL)
    assert st == B.KDA_ERR_UNSUPPORTED


def _prefill_gated(lib, fn="kda_prefill_gated", **over):
    a = dict(q=0x10000, k=0x20000, v=0x30000, z=0x40000, A=0xa0000, beta=0x50000, cu=0x60000, N=1, T=4, H=2,
             dk=128, dv=128, dtype=1, odtype=0, gmin=-5.0, scale=1.0, init=NULL, out=0x70000, fin=0x80000,
             stream=NULL)
    a.update(over)
    return getattr(lib, fn)(a["q"], a["k"], a["v"], a["z"], a["A"], a["beta"], a["cu"], a["N"], a["T"], a["H"],
                            a["dk"], a["dv"], a["dtype"], a["odtype"], a["gmin"], a["scale"], a["init"], a["out"],
                            a["fin"], a["stream"])


@pytest.mark.parametrize("fn", ["kda_prefill_gated", "kda_prefill_gated_recurrent"])
@pytest.mark.parametrize("over,expect", [
    (dict(z=NULL), B.KDA_ERR_INVALID_ARG),
    (dict(A=NULL), B.KDA_ERR_INVALID_ARG),
    (dict(A=0xa0002), B.KDA_ERR_INVALID_ARG),          # misaligned A_log
    (dict(z=0x40008), B.KDA_ERR_INVALID_ARG),          # misaligned z
    (dict(gmin=0.5), B.KDA_ERR_INVALID_ARG),           # g_min must be <= 0
    (dict(gmin=float("nan")), B.KDA_ERR_INVALID_ARG),
    (dict(gmin=float("-inf")), B.KDA_ERR_INVALID_ARG),
    (dict(out=0x40000), B.KDA_ERR_INVALID_ARG),        # output aliases z
    (dict(fin=0xa0000), B.KDA_ERR_INVALID_ARG),        # final state aliases A_log
    (dict(dk=129), B.KDA_ERR_UNSUPPORTED),
])
def test_prefill_gated_rejects(lib, fn, over, expect):
    assert _prefill_gated(lib, fn, **over) == expect


def test_prefill_gated_accepts_empty_work(lib):
    assert _prefill_gated(lib, N=0, T=0, q=NULL, k=NULL, v=NULL, z=NULL, beta=NULL, out=NULL, fin=NULL) == B.KDA_OK


@pytest.mark.parametrize("over,expect", [
    (dict(z=NULL), B.KDA_ERR_INVALID_ARG),
    (dict(A=NULL), B.KDA_ERR_INVALID_ARG),
    (dict(gmin=1.0), B.KDA_ERR_INVALID_ARG),
    (dict(state=NULL), B.KDA_ERR_INVALID_ARG),
    (dict(dv=6), B.KDA_ERR_UNSUPPORTED),
])
def test_decode_gated_rejects(lib, over, expect):
    a = dict(q=0x10000, k=0x20000, v=0x30000, z=0x40000, A=0xa0000, beta=0x50000, state=0x90000, out=0x70000, B=2,
             H=2, dk=128, dv=128, dtype=1, odtype=0, gmin=-5.0)
    a.update(over)
    st = lib.kda_decode_gated(a["q"], a["k"], a["v"], a["z"], a["A"], a["beta"], a["state"], a["out"], a["B"],
                              a["H"], a["dk"], a["dv"], a["dtype"], a["odtype"], a["gmin"], 1.0, NULL)
    assert st == expect


def _prefill_ex(lib, **over):
    """A parameter block with fake device addresses: validation must reject before any CUDA call."""
    f = dict(struct_size=ctypes.sizeof(B.PrefillParams), in_dtype=1, out_dtype=0, decay_form=0, num_seqs=1, H=2,
             d_k=128, d_v=128, total_tokens=4, q=0x10000, k=0x20000, v=0x30000, decay=0x40000, A_log=None,
             beta=0x50000, cu_seqlens=0x60000, init_state=None, out_gate=0xb0000, norm_weight=0xc0000,
             out=0x70000, final_state=0x80000, decay_bound=-5.0, scale=1.0, norm_eps=1e-6, force_recurrent=0,
             workspace=None, workspace_bytes=0)
    f.update(over)
    return lib.kda_prefill_ex(ctypes.byref(B.PrefillParams(**f)), NULL)


@pytest.mark.parametrize("over,expect", [
    (dict(struct_size=148), B.KDA_ERR_INVALID_ARG),                 # not this library's struct
    (dict(decay_form=2), B.KDA_ERR_INVALID_ARG),
    (dict(A_log=0xa0000), B.KDA_ERR_INVALID_ARG),                   # A_log with the clamped form
    (dict(decay_form=1), B.KDA_ERR_INVALID_ARG),                    # gated form without A_log
    (dict(decay_form=1, A_log=0xa0000, decay_bound=1.0), B.KDA_ERR_INVALID_ARG),
    (dict(decay_form=2), B.KDA_ERR_INVALID_ARG),                    # unbounded form without A_log
    (dict(decay_form=2, A_log=0xa0002), B.KDA_ERR_INVALID_ARG),     # misaligned A_log
    (dict(decay_form=3, A_log=0xa0000), B.KDA_ERR_INVALID_ARG),
    (dict(out_gate=None), B.KDA_ERR_INVALID_ARG),                   # a weight without gate logits
    (dict(norm_eps=float("nan")), B.KDA_ERR_INVALID_ARG),
    (dict(norm_eps=-1.0), B.KDA_ERR_INVALID_ARG),
    (dict(norm_eps=float("inf")), B.KDA_ERR_INVALID_ARG),
    (dict(out_gate=0xb0008), B.KDA_ERR_INVALID_ARG),                # misaligned gate logits
    (dict(norm_weight=0xc0002), B.KDA_ERR_INVALID_ARG),
    (dict(out=0xb0000), B.KDA_ERR_INVALID_ARG),                     # output over the gate logits
    (dict(final_state=0xc0000), B.KDA_ERR_INVALID_ARG),             # final state over the weight
    (dict(in_dtype=5), B.KDA_ERR_INVALID_ARG),
    (dict(d_v=129), B.KDA_ERR_UNSUPPORTED),
    (dict(q=None), B.KDA_ERR_INVALID_ARG),
    (dict(workspace=0x1000000), B.KDA_ERR_INVALID_ARG),               # workspace without bytes
    (dict(workspace=0xb0000, workspace_bytes=64), B.KDA_ERR_INVALID_ARG),  # workspace over the gate logits
])
def test_prefill_ex_rejects(lib, over, expect):
    assert _prefill_ex(lib, **over) == expect


def test_prefill_ex_accepts_empty_work(lib):
    assert _prefill_ex(lib, num_seqs=0, total_tokens=0, q=None, k=None, v=None, decay=None, beta=None, out=None,
                       final_state=None, out_gate=None, norm_weight=None) == B.KDA_OK
    assert _prefill_ex(lib, num_seqs=0, total_tokens=0, decay_form=1, A_log=0xa0000) == B.KDA_OK
    assert _prefill_ex(lib, num_seqs=0, total_tokens=0, decay_form=2, A_log=0xa0000, decay_bound=7.0) == B.KDA_OK


def _decode_ex(lib, **over):
    f = dict(struct_size=ctypes.sizeof(B.DecodeParams), in_dtype=1, out_dtype=0, decay_form=0, B=2, H=2, d_k=128,
             d_v=128, q=0x10000, k=0x20000, v=0x30000, decay=0x40000, A_log=None, beta=0x50000, state=0x1000000,
             out_gate=0xb0000, norm_weight=None, out=0x70000, conv_weight=None, conv_state=None, decay_bound=-5.0,
             scale=1.0, norm_eps=1e-6, l2_eps=1e-6)
    f.update(over)
    return lib.kda_decode_ex(ctypes.byref(B.DecodeParams(**f)), NULL)


@pytest.mark.parametrize("over,expect", [
    (dict(struct_size=0), B.KDA_ERR_INVALID_ARG),
    (dict(decay_form=7), B.KDA_ERR_INVALID_ARG),
    (dict(A_log=0xa0000), B.KDA_ERR_INVALID_ARG),
    (dict(decay_form=1, A_log=0xa0000, decay_bound=float("nan")), B.KDA_ERR_INVALID_ARG),
    (dict(out_gate=None, norm_weight=0xc0000), B.KDA_ERR_INVALID_ARG),
    (dict(norm_eps=-0.5), B.KDA_ERR_INVALID_ARG),
    (dict(out_gate=0xb0004), B.KDA_ERR_INVALID_ARG),
    (dict(out=0xb0000), B.KDA_ERR_INVALID_ARG),                     # output over the gate logits
    (dict(d_v=6), B.KDA_ERR_UNSUPPORTED),
    (dict(state=None), B.KDA_ERR_INVALID_ARG),
    (dict(conv_weight=0xd0000), B.KDA_ERR_INVALID_ARG),             # conv weights without a state
    (dict(conv_state=0xe0000), B.KDA_ERR_INVALID_ARG),              # a state without weights
    (dict(conv_state=0xe0000, conv_weight=0xd0000, l2_eps=float("nan")), B.KDA_ERR_INVALID_ARG),
    (dict(conv_state=0xe0008, conv_weight=0xd0000), B.KDA_ERR_INVALID_ARG),
    (dict(conv_state=0x1000000 + 4096, conv_weight=0xd0000), B.KDA_ERR_INVALID_ARG),  # inside the state
    (dict(conv_state=0x20000, conv_weight=0xd0000), B.KDA_ERR_INVALID_ARG),         # over k
    (dict(state=0xb0000 - 4096), B.KDA_ERR_INVALID_ARG),                            # state into the gate logits
    (dict(out=0x1000000 + 65536), B.KDA_ERR_INVALID_ARG),                           # out inside the state
])
def test_decode_ex_rejects(lib, over, expect):
    assert _decode_ex(lib, **over) == expect


def test_parameter_blocks_have_the_header_layout():
    """The ctypes mirrors add up to the sizes the header's field order gives on LP64 (no padding)."""
    assert ctypes.sizeof(B.PrefillParams) == 16 + 16 + 8 + 12 * 8 + 16 + 16
    assert ctypes.sizeof(B.DecodeParams) == 16 + 16 + 12 * 8 + 16


def _prologue(lib, **over):
    a = dict(q_raw=0x10000, k_raw=0x20000, v_raw=0x30000, w=0x40000, cu=0x60000, N=1, T=4, H=2, dk=128, dv=128,
             dtype=1, init=None, eps=1e-6, q=0x70000, k=0x80000, v=0x90000, fin=0xa0000)
    a.update(over)
    return lib.kda_prologue(a["q_raw"], a["k_raw"], a["v_raw"], a["w"], a["cu"], a["N"], a["T"], a["H"], a["dk"],
                            a["dv"], a["dtype"], a["init"], a["eps"], a["q"], a["k"], a["v"], a["fin"], NULL)


@pytest.mark.parametrize("over,expect", [
    (dict(w=None), B.KDA_ERR_INVALID_ARG),
    (dict(cu=None), B.KDA_ERR_INVALID_ARG),
    (dict(q=None), B.KDA_ERR_INVALID_ARG),
    (dict(v_raw=0x30008), B.KDA_ERR_INVALID_ARG),
    (dict(dtype=3), B.KDA_ERR_INVALID_ARG),
    (dict(eps=-1.0), B.KDA_ERR_INVALID_ARG),
    (dict(eps=float("inf")), B.KDA_ERR_INVALID_ARG),
    (dict(dk=200), B.KDA_ERR_UNSUPPORTED),
    (dict(H=70000), B.KDA_ERR_UNSUPPORTED),
    (dict(N=0), B.KDA_ERR_INVALID_ARG),                     # tokens without a sequence
    (dict(q=0x10000), B.KDA_ERR_INVALID_ARG),               # output over an input
    (dict(k=0x70000), B.KDA_ERR_INVALID_ARG),               # two outputs overlap
    (dict(init=0xb0000, fin=0xb0000), B.KDA_ERR_INVALID_ARG),  # final state over the initial one
])
def test_prologue_rejects(lib, over, expect):
    assert _prologue(lib, **over) == expect


def test_prologue_accepts_empty_work(lib):
    assert _prologue(lib, N=0, T=0, q_raw=None, k_raw=None, v_raw=None, q=None, k=None, v=None, fin=None) == B.KDA_OK


def test_wait_selftest_rejects_bad_status_pointer(lib):
    assert lib.kda_selftest_wait_timeout(NULL, NULL) == B.KDA_ERR_INVALID_ARG
    assert lib.kda_selftest_wait_timeout(0x1002, NULL) == B.KDA_ERR_INVALID_ARG
