"""CPU pins of the oracle's input prologue: ShortConv (4 taps, causal, depthwise)
-> Swish on q, k, v -> L2 norm on q and k (Kimi K3 -- Architecture Notes, section
1.1; kernel size 4 from the visualiser page "Kimi K3").

The pins are values worked out by hand (decimal-digit taps make every tap's
contribution readable in the result), Swish at points where it has a closed form,
the unit norm of q and k, and properties of a causal per-sequence window: a delayed
copy, the reset at each sequence start, the carried convolution state, and packed
sequences equal to separate calls. Each planted mistake must fail one of them.
"""

import math

import numpy as np
import pytest

from oracle.prologue import PROLOGUE_MUTATIONS, kda_prologue, short_conv


def _taps(H, C, taps):
    w = np.zeros((H, C, 4))
    w[:, :, :] = np.asarray(taps, dtype=np.float64)
    return w


def pin_decimal_taps(mut):
    """One channel, x = 1..5, taps (1, 10, 100, 1000) on (t-3, t-2, t-1, t): the result's digits
    are the window, newest first. With the state (7, 8, 9) before the sequence the first
    three results read 1987, 2198, 3219."""
    x = np.arange(1.0, 6.0).reshape(5, 1, 1)
    w = _taps(1, 1, [1, 10, 100, 1000])
    y, fin = short_conv(x, w, [0, 5], mutation=mut)
    assert np.array_equal(y[:, 0, 0], [1000, 2100, 3210, 4321, 5432]), y[:, 0, 0]
    assert np.array_equal(fin[0, 0, :, 0], [3, 4, 5])
    st = np.array([7.0, 8.0, 9.0]).reshape(1, 1, 3, 1)
    y, _ = short_conv(x, w, [0, 5], state=st, mutation=mut)
    assert np.array_equal(y[:, 0, 0], [1987, 2198, 3219, 4321, 5432]), y[:, 0, 0]


def pin_sequence_reset_and_state(mut):
    """Packed sequences [4, 2, 0, 3]: each window restarts at its sequence start and reads the
    sequence's own state; the final state holds the last three inputs, shifted in from the
    state when the sequence is shorter than three; an empty sequence passes its state on."""
    rng = np.random.default_rng(7)
    lens = [4, 2, 0, 3]
    cu = np.concatenate([[0], np.cumsum(lens)])
    x = rng.standard_normal((9, 2, 3))
    w = rng.standard_normal((2, 3, 4))
    st = rng.standard_normal((4, 2, 3, 3))
    y, fin = short_conv(x, w, cu, state=st, mutation=mut)
    for n in range(4):
        yn, fn = short_conv(x[cu[n]:cu[n + 1]], w, [0, lens[n]], state=st[n:n + 1], mutation=mut)
        assert np.allclose(y[cu[n]:cu[n + 1]], yn, rtol=0, atol=1e-14)
        assert np.allclose(fin[n], fn[0], rtol=0, atol=0)
    assert np.array_equal(fin[1, :, 0], st[1, :, 2]) and np.array_equal(fin[1, :, 1:], x[4:6].transpose(1, 0, 2))
    assert np.array_equal(fin[2], st[2])
    # a delay of three: y_t = x_{t-3}, from the state for the first three tokens
    w3 = _taps(2, 3, [1, 0, 0, 0])
    y, _ = short_conv(x, w3, cu, state=st, mutation=mut)
    assert np.array_equal(y[0:3], st[0].transpose(1, 0, 2)) and np.array_equal(y[3], x[0])


def pin_swish_points(mut):
    """Identity taps: q, k, v see x itself. Swish(x) = x Sigmoid(x): 0 at 0, (3/4) ln 3 at ln 3,
    -(1/4) ln 3 at -ln 3. v keeps Swish(x); q and k are Swish(x) / |Swish(x)|."""
    H, dk, dv = 1, 2, 3
    ln3 = math.log(3.0)
    x = np.array([[[ln3, -ln3, 0.0, ln3, -ln3, 0.0, ln3]]])  # q (2), k (2), v (3)
    w = _taps(H, 2 * dk + dv, [0, 0, 0, 1])
    q, k, v, _ = kda_prologue(x[..., :2], x[..., 2:4], x[..., 4:], w, [0, 1], eps=0.0, mutation=mut)
    assert np.allclose(v[0, 0], [-0.25 * ln3, 0.0, 0.75 * ln3], rtol=1e-14, atol=1e-15), v
    sq = np.array([0.75 * ln3, -0.25 * ln3])
    assert np.allclose(q[0, 0], sq / np.linalg.norm(sq), rtol=1e-14), q
    sk = np.array([0.0, 0.75 * ln3])
    assert np.allclose(k[0, 0], sk / np.linalg.norm(sk), rtol=1e-14), k


def pin_unit_norm(mut):
    """q and k rows have norm 1 (to within eps / |Swish|^2); v rows do not."""
    rng = np.random.default_rng(8)
    T, H, d = 12, 3, 8
    q0, k0, v0 = (rng.standard_normal((T, H, d)) for _ in range(3))
    w = rng.standard_normal((H, 3 * d, 4))
    q, k, v, _ = kda_prologue(q0, k0, v0, w, [0, 5, 12], eps=1e-12, mutation=mut)
    assert np.allclose(np.linalg.norm(q, axis=-1), 1.0, atol=1e-9)
    assert np.allclose(np.linalg.norm(k, axis=-1), 1.0, atol=1e-9)
    assert not np.allclose(np.linalg.norm(v, axis=-1), 1.0, atol=1e-3)


def pin_swish_sign(mut):
    """Swish(x) < 0 exactly where x < 0, and Swish(x) >= -0.2785 (its minimum)."""
    rng = np.random.default_rng(9)
    x = 3.0 * rng.standard_normal((7, 2, 5))
    w = _taps(2, 15, [0, 0, 0, 1])
    _, _, v, _ = kda_prologue(np.zeros((7, 2, 5)), np.zeros((7, 2, 5)), x, w, [0, 7], mutation=mut)
    assert np.array_equal(v < 0, x < 0) and v.min() >= -0.2785


PINS = [pin_decimal_taps, pin_sequence_reset_and_state, pin_swish_points, pin_unit_norm, pin_swish_sign]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_prologue_pins(pin):
    pin(None)


@pytest.mark.parametrize("mutation", PROLOGUE_MUTATIONS)
def test_planted_prologue_mistake_is_caught(mutation):
    failed = []
    for pin in PINS:
        try:
            pin(mutation)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {mutation!r}"


def test_rejects_bad_weight_shape():
    with pytest.raises(ValueError):
        kda_prologue(np.zeros((2, 1, 4)), np.zeros((2, 1, 4)), np.zeros((2, 1, 4)), np.zeros((1, 12, 3)), [0, 2])
