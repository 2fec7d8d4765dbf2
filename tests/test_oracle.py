"""CPU tests that pin the oracle to the definition and to mathematics, not to itself.

Definition: Kimi K3 -- Architecture Notes, section 1.1 (the KDA recurrence) and
section 1.2 (the lower-bounded decay). No worked numeric example exists on the
pages, so the pins are exact brute force, closed forms, invariants, agreement
between independent restatements, and planted mistakes that must be caught.
"""

import json
import os
from fractions import Fraction

import numpy as np
import pytest

import pins
from oracle import MUTATIONS, chunk_quantities, kda_chunked, kda_exact, kda_recurrent, kda_recurrent_mutant

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def run_recurrent(q, k, v, g, b, cu, lower_bound=-5.0, init_state=None):
    return kda_recurrent(q, k, v, g, b, cu, lower_bound=lower_bound, init_state=init_state, num_threads=2)


def make_chunked(chunk):
    def run(q, k, v, g, b, cu, lower_bound=-5.0, init_state=None):
        return kda_chunked(q, k, v, g, b, cu, chunk=chunk, lower_bound=lower_bound, init_state=init_state)
    return run


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_recurrent_oracle_pins(pin):
    pin(run_recurrent)


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
@pytest.mark.parametrize("chunk", [1, 4])
def test_chunked_oracle_pins(pin, chunk):
    pin(make_chunked(chunk))


@pytest.mark.parametrize("name,mut", sorted(MUTATIONS.items()))
def test_planted_mistakes_are_caught(name, mut):
    """Each plausible mistake planted in the C oracle fails at least one pin."""
    def run(q, k, v, g, b, cu, lower_bound=-5.0, init_state=None):
        return kda_recurrent_mutant(q, k, v, g, b, cu, mutation=mut, lower_bound=lower_bound,
                                    init_state=init_state, num_threads=1)
    failures = []
    for pin in pins.ALL_PINS:
        try:
            pin(run)
        except AssertionError:
            failures.append(pin.__name__)
        except RuntimeError:
            pass  # shapes a mutant cannot run (value-axis decay needs d_k == d_v)
    assert failures, f"mutation {name} passed every pin"


def _random_problem(rng, lengths, H, dk, dv, strong=False):
    T = sum(lengths)
    q = rng.standard_normal((T, H, dk)); q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((T, H, dk)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    if strong:
        g = -5.0 + 0.25 * rng.standard_normal((T, H, dk))
    else:
        g = -np.logaddexp(0.0, rng.standard_normal((T, H, dk)))
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    S0 = 0.02 * rng.standard_normal((len(lengths), H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    return q, k, v, g, b, cu, S0


@pytest.mark.parametrize("chunk", [1, 16, 64])
@pytest.mark.parametrize("strong", [False, True])
def test_recurrent_matches_chunked(chunk, strong):
    """The token-by-token and chunkwise restatements agree to fp64 round-off,
    with ragged tails, an empty and a length-1 sequence, and strong decay."""
    rng = np.random.default_rng(100 + chunk)
    lengths = [70, 0, 1, 130, 17]
    q, k, v, g, b, cu, S0 = _random_problem(rng, lengths, 2, 16, 12, strong=strong)
    o_r, f_r = kda_recurrent(q, k, v, g, b, cu, init_state=S0, num_threads=2)
    o_c, f_c = kda_chunked(q, k, v, g, b, cu, chunk=chunk, init_state=S0)
    assert pins.rel_err(o_c, o_r) < 1e-12
    assert pins.rel_err(f_c, f_r) < 1e-12


def test_ut_inverse_is_inverse():
    """(I + A) T = I for every chunk; T is unit lower triangular."""
    rng = np.random.default_rng(11)
    q, k, v, g, b, cu, _ = _random_problem(rng, [64], 1, 32, 8)
    g = np.maximum(g, -5.0)
    cq = chunk_quantities(q[:, 0], k[:, 0], v[:, 0], g[:, 0], b[:, 0])
    L = q.shape[0]
    assert np.max(np.abs((np.eye(L) + cq["A"]) @ cq["T"] - np.eye(L))) < 1e-12
    assert np.allclose(np.triu(cq["T"], 1), 0.0) and np.allclose(np.diag(cq["T"]), 1.0)


def test_toy_form_differs_when_decaying():
    """Negative control. The llm-vis 'Kimi Delta Attention (KDA)' block states
    S_t = Diag(a) S_{t-1} + b (v - S_{t-1} k) k^T on a value-major state, which
    predicts with the undecayed state. It agrees with the architecture-notes
    form when alpha = 1 and must differ from the oracle when alpha < 1."""
    rng = np.random.default_rng(12)
    T, d = 9, 6
    q, k, v, g, b, cu, _ = _random_problem(rng, [T], 1, d, d)

    def toy(gv):
        S = np.zeros((d, d))  # value-major: S @ k is a value vector
        outs = []
        for t in range(T):
            a = np.exp(gv[t, 0])
            S = a[:, None] * S + b[t, 0] * np.outer(v[t, 0] - S @ k[t, 0], k[t, 0])
            outs.append(S @ q[t, 0])
        return np.array(outs)

    zero = np.zeros_like(g)
    o_or, _ = kda_recurrent(q, k, v, zero, b, cu, num_threads=1)
    assert pins.rel_err(toy(zero), o_or[:, 0]) < 1e-13
    o_or, _ = kda_recurrent(q, k, v, g, b, cu, num_threads=1)
    assert pins.rel_err(toy(g), o_or[:, 0]) > 1e-3


def test_decay_bound_arithmetic_printed_on_page():
    """Kimi K3 -- Architecture Notes, section 1.2 prints g_min = -5, 16-token
    tiles, a bound of e^80 on the reciprocal rescaling, and says it stays
    within bf16 range; check the arithmetic the chunked kernels rely on."""
    with open(os.path.join(GOLDEN, "decay_bound.json")) as fh:
        gold = json.load(fh)
    g_min, tile = gold["g_min"], gold["tile_tokens"]
    assert g_min * tile == -gold["log_bound"]
    bf16_max = float.fromhex("0x1.fep127")  # largest finite bf16 (= 3.39e38)
    f32_max = float.fromhex("0x1.fffffep127")
    assert gold["log_bound"] < np.log(bf16_max) < np.log(f32_max)
    assert abs(np.exp(g_min) - gold["alpha_min_approx"]) < 0.05e-3
    # a 64-token chunk with one reference point would not fit (4 tiles x 80 > 88.7)
    assert 4 * gold["log_bound"] > np.log(f32_max)


def test_golden_exact_fixture():
    """The C oracle reproduces the stored exact rational results (written by
    tests/golden/make_golden.py, which calls only oracle.exact)."""
    with open(os.path.join(GOLDEN, "kda_exact_tiny.json")) as fh:
        gold = json.load(fh)
    for case in gold["cases"]:
        fr = lambda m: np.array([[float(Fraction(x)) for x in row] for row in m])
        q, k, v, alpha = fr(case["q"]), fr(case["k"]), fr(case["v"]), fr(case["alpha"])
        beta = np.array([float(Fraction(x)) for x in case["beta"]])
        S0 = fr(case["S0"])
        out, fin = kda_recurrent(q[:, None], k[:, None], v[:, None], np.log(alpha)[:, None],
                                 beta[:, None], [0, q.shape[0]], lower_bound=pins.NO_CLAMP,
                                 init_state=S0[None, None], num_threads=1)
        assert pins.rel_err(out[:, 0], fr(case["o"])) < 1e-13
        assert pins.rel_err(fin[0, 0], fr(case["S_T"])) < 1e-13
        # and the fixture is still what the exact brute force produces
        o_ex, S_ex = kda_exact(case["q"], case["k"], case["v"], case["alpha"], case["beta"], case["S0"])
        assert [[str(x) for x in r] for r in o_ex] == case["o"]
        assert [[str(x) for x in r] for r in S_ex] == case["S_T"]


def test_nan_log_alpha_propagates():
    """A NaN log-decay is not clamped away: the clamp is g < lb ? lb : g."""
    q = np.ones((1, 1, 2)) / np.sqrt(2.0)
    g = np.array([[[np.nan, -1.0]]])
    out, fin = kda_recurrent(q, q, np.ones((1, 1, 2)), g, np.full((1, 1), 0.5), [0, 1],
                             init_state=np.ones((1, 1, 2, 2)), num_threads=1)
    assert np.isnan(fin[0, 0, 0]).all() and np.isnan(out).all()


def test_oracle_rejects_bad_cu_seqlens():
    q = np.zeros((3, 1, 2))
    with pytest.raises(ValueError):
        kda_recurrent(q, q, q, q, np.zeros((3, 1)), [0, 2], num_threads=1)
    with pytest.raises(RuntimeError):
        kda_recurrent(q, q, q, q, np.zeros((3, 1)), [0, 2, 1, 3], num_threads=1)
