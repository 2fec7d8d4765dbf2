"""CPU pins of the oracle's output gate with head-wise RMSNorm,
out = Sigmoid(r) * w * o / sqrt(mean(o^2) + eps) over the d_v channels of each
(token, head) (Kimi K3 -- Architecture Notes, section 1.3 "Full-rank output gate").

The pins are values worked out by hand for small vectors, and properties the
definition fixes whatever the numbers: Sigmoid(r) + Sigmoid(-r) = 1, the RMS of
the normalised vector is 1, invariance to a positive rescaling of o, oddness in
o, independence of other heads and other tokens, and the eps limit for a tiny o.
Each planted mistake must fail at least one of them.
"""

import math

import numpy as np
import pytest

from oracle.epilogue import EPILOGUE_MUTATIONS, output_gate_rmsnorm


def _run(mutation):
    return lambda o, r, w=None, eps=1e-6: output_gate_rmsnorm(o, r, w, eps, mutation=mutation)


def pin_hand_values(f):
    """Worked by hand. o = (3, 4): mean of squares 12.5, so o / sqrt(12.5) = (0.6 sqrt 2, 0.8 sqrt 2).
    Gate logits (0, ln 3): Sigmoid = (1/2, 3/4). Weight (2, 1/2)."""
    o = np.array([[[3.0, 4.0]]])
    r = np.array([[[0.0, math.log(3.0)]]])
    w = np.array([2.0, 0.5])
    y = f(o, r, w, 0.0)
    expect = np.array([0.5 * 2.0 * 0.6 * math.sqrt(2.0), 0.75 * 0.5 * 0.8 * math.sqrt(2.0)])
    assert np.allclose(y[0, 0], expect, rtol=1e-14, atol=0), (y, expect)
    # o = (1, -2, 3, -4): mean of squares 7.5; eps = 0.5 makes the divisor sqrt(8) = 2 sqrt 2
    o = np.array([[[1.0, -2.0, 3.0, -4.0]]])
    r = np.array([[[0.0, 0.0, -math.log(3.0), math.log(3.0)]]])
    y = f(o, r, None, 0.5)
    expect = np.array([0.5, -1.0, 0.75, -3.0]) / (2.0 * math.sqrt(2.0))
    assert np.allclose(y[0, 0], expect, rtol=1e-14, atol=0), (y, expect)


def pin_unit_rms(f):
    """Saturated gate (r = 40: Sigmoid = 1 to within 5e-18), w = 1, eps = 0: every (token, head)
    row of the result has RMS exactly 1."""
    rng = np.random.default_rng(3)
    o = rng.standard_normal((5, 3, 16)) * rng.uniform(0.01, 100.0, (5, 3, 1))
    y = f(o, np.full_like(o, 40.0), None, 0.0)
    rms = np.sqrt(np.mean(y * y, axis=-1))
    assert np.allclose(rms, 1.0, rtol=1e-13, atol=0), rms


def pin_gate_complement(f):
    """Sigmoid(r) + Sigmoid(-r) = 1, and r = 0 halves: f(o, r) + f(o, -r) = 2 f(o, 0)."""
    rng = np.random.default_rng(4)
    o = rng.standard_normal((4, 2, 8))
    r = 3.0 * rng.standard_normal(o.shape)
    w = rng.uniform(0.5, 2.0, 8)
    a = f(o, r, w) + f(o, -r, w)
    b = 2.0 * f(o, np.zeros_like(r), w)
    assert np.allclose(a, b, rtol=1e-13, atol=1e-15)
    # a saturated gate (Sigmoid(40) = 1 - 4e-18) passes w * RMSNorm(o) = 2 f(o, 0) through
    assert np.allclose(f(o, np.full_like(r, 40.0), w), b, rtol=1e-15, atol=0)


def pin_scale_and_sign(f):
    """eps = 0: f(c o) = f(o) for c > 0, f(-o) = -f(o)."""
    rng = np.random.default_rng(5)
    o = rng.standard_normal((6, 2, 8))
    r = rng.standard_normal(o.shape)
    y = f(o, r, None, 0.0)
    for c in (1e-3, 7.0, 1e4):
        assert np.allclose(f(c * o, r, None, 0.0), y, rtol=1e-12, atol=0)
    assert np.allclose(f(-o, r, None, 0.0), -y, rtol=1e-15, atol=0)


def pin_head_and_token_independence(f):
    """Changing one head (or one token) leaves every other head's (token's) result unchanged."""
    rng = np.random.default_rng(6)
    o = rng.standard_normal((7, 3, 8))
    r = rng.standard_normal(o.shape)
    y = f(o, r)
    o2 = o.copy()
    o2[:, 1] *= 50.0
    y2 = f(o2, r)
    assert np.array_equal(y2[:, 0], y[:, 0]) and np.array_equal(y2[:, 2], y[:, 2])
    o3 = o.copy()
    o3[2] *= 50.0
    y3 = f(o3, r)
    assert np.array_equal(np.delete(y3, 2, axis=0), np.delete(y, 2, axis=0))


def pin_eps_limit(f):
    """|o|^2 << eps: the divisor tends to sqrt(eps), so f(o) -> Sigmoid(r) w o / sqrt(eps); o = 0 gives 0."""
    o = np.array([[[1e-9, -2e-9, 3e-9, 0.0]]])
    r = np.zeros_like(o)
    y = f(o, r, None, 1e-2)
    assert np.allclose(y, 0.5 * o / 0.1, rtol=1e-12, atol=0), y
    assert np.array_equal(f(np.zeros((2, 1, 4)), np.ones((2, 1, 4)), None, 1e-6), np.zeros((2, 1, 4)))


PINS = [pin_hand_values, pin_unit_rms, pin_gate_complement, pin_scale_and_sign,
        pin_head_and_token_independence, pin_eps_limit]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_epilogue_pins(pin):
    pin(_run(None))


@pytest.mark.parametrize("mutation", EPILOGUE_MUTATIONS)
def test_planted_epilogue_mistake_is_caught(mutation):
    failed = []
    for pin in PINS:
        try:
            pin(_run(mutation))
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {mutation!r}"


def test_rejects_bad_shapes():
    with pytest.raises(ValueError):
        output_gate_rmsnorm(np.zeros((2, 1, 4)), np.zeros((2, 1, 3)))
    with pytest.raises(ValueError):
        output_gate_rmsnorm(np.zeros((2, 1, 4)), np.zeros((2, 1, 4)), np.ones(3))
