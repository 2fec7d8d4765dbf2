"""CPU pins of the oracle's gated log-decay, g = g_min * Sigmoid(e^{A_h} z)
(Kimi K3 -- Architecture Notes, section 1.2, the K3 row of the mapping table).

Each pin compares the gated oracle with the clamped one on inputs where the
gate's value is fixed by mathematics alone: Sigmoid(0) = 1/2 for every A_h, the
saturated limits of very large |e^{A_h} z|, the strict bounds g in (g_min, 0),
and the monotonicity in z. Planted mistakes in the gate (A_h where e^{A_h}
belongs, the unbounded Softplus map of the earlier models, a flipped sign) must
each fail one of them.
"""

import numpy as np
import pytest

from oracle import GATE_MUTATIONS, kda_recurrent, kda_recurrent_gated

G_MIN = -5.0


def _problem(rng, T, H, dk, dv):
    q = rng.standard_normal((T, H, dk)); q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((T, H, dk)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    S0 = 0.02 * rng.standard_normal((2, H, dk, dv))
    cu = np.array([0, T // 3, T])
    return q, k, v, b, cu, S0


def _gated(mutation):
    def run(q, k, v, z, A, b, cu, S0):
        return kda_recurrent_gated(q, k, v, z, A, b, cu, g_min=G_MIN, init_state=S0, num_threads=2,
                                   mutation=mutation)
    return run


def _clamped(q, k, v, g, b, cu, S0):
    return kda_recurrent(q, k, v, g, b, cu, lower_bound=G_MIN, init_state=S0, num_threads=2)


def _close(a, b, tol):
    for x, y in zip(a, b):
        scale = max(float(np.abs(y).max()), 1e-300)
        assert float(np.abs(x - y).max()) <= tol * scale, float(np.abs(x - y).max()) / scale


def pin_zero_logit(run):
    """z = 0: Sigmoid(e^{A_h} 0) = 1/2 for any A_h, so g = g_min / 2 exactly."""
    rng = np.random.default_rng(20)
    q, k, v, b, cu, S0 = _problem(rng, 23, 3, 8, 5)
    z = np.zeros_like(q)
    A = np.array([-3.0, 0.0, 4.0])
    _close(run(q, k, v, z, A, b, cu, S0), _clamped(q, k, v, np.full_like(q, G_MIN / 2), b, cu, S0), 1e-15)


def pin_saturated_limits(run):
    """e^{A_h} z -> +inf gives g = g_min, -> -inf gives g = 0 (alpha = 1), both exactly in fp64."""
    rng = np.random.default_rng(21)
    q, k, v, b, cu, S0 = _problem(rng, 19, 2, 6, 7)
    z = np.where(rng.standard_normal(q.shape) > 0, 1.0e3, -1.0e3)
    A = np.array([0.0, 1.0])
    g = np.where(z > 0, G_MIN, 0.0)
    _close(run(q, k, v, z, A, b, cu, S0), _clamped(q, k, v, g, b, cu, S0), 1e-15)


def pin_per_head_scale(run):
    """Head 0 with e^{A_0} ~ 2e-22 sits at the midpoint g_min/2; head 1 with e^{A_1} ~ 2.2e4
    and |z| = 0.1 saturates to g_min or 0 by the sign of z: A_h belongs to its own head and
    enters through e^{A_h}."""
    rng = np.random.default_rng(22)
    q, k, v, b, cu, S0 = _problem(rng, 21, 2, 6, 6)
    z = 0.1 * np.sign(rng.standard_normal(q.shape))
    A = np.array([-50.0, 10.0])
    g = np.empty_like(q)
    g[:, 0] = G_MIN / 2
    g[:, 1] = np.where(z[:, 1] > 0, G_MIN, 0.0)
    _close(run(q, k, v, z, A, b, cu, S0), _clamped(q, k, v, g, b, cu, S0), 1e-12)


def pin_bounds_and_monotone(run):
    """With beta = 0 and d_k = d_v = 1 one step gives S_1 = alpha S_0: every alpha lies in
    (e^{g_min}, 1) and decreases as z grows (fixed A_h)."""
    T, H = 1, 64
    z = np.linspace(-4.0, 4.0, H).reshape(1, H, 1)
    A = np.full(H, 0.3)
    q = np.ones((T, H, 1)); k = np.ones((T, H, 1)); v = np.zeros((T, H, 1))
    b = np.zeros((T, H))
    S0 = np.ones((1, H, 1, 1))
    _, fin = run(q, k, v, z, A, b, np.array([0, T]), S0)
    alpha = fin[0, :, 0, 0]
    assert np.all(alpha > np.exp(G_MIN)) and np.all(alpha < 1.0)
    assert np.all(np.diff(alpha) < 0)


GATE_PINS = [pin_zero_logit, pin_saturated_limits, pin_per_head_scale, pin_bounds_and_monotone]


@pytest.mark.parametrize("pin", GATE_PINS, ids=lambda p: p.__name__)
def test_gated_oracle_pins(pin):
    pin(_gated(0))


@pytest.mark.parametrize("name,mut", sorted(GATE_MUTATIONS.items()))
def test_gate_planted_mistakes_are_caught(name, mut):
    failures = []
    for pin in GATE_PINS:
        try:
            pin(_gated(mut))
        except AssertionError:
            failures.append(pin.__name__)
    assert failures, f"gate mutation {name} passed every pin"


def test_gated_oracle_reads_bf16_logits():
    """z given as bf16 bits is read exactly: the same values as float32 inputs."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(23)
    q, k, v, b, cu, S0 = _problem(rng, 9, 2, 4, 3)
    z32 = torch.tensor(rng.standard_normal(q.shape), dtype=torch.float32).bfloat16()
    A = np.array([0.2, -0.4])
    a = kda_recurrent_gated(q, k, v, z32, A, b, cu, g_min=G_MIN, init_state=S0)
    c = kda_recurrent_gated(q, k, v, z32.float().numpy(), A, b, cu, g_min=G_MIN, init_state=S0)
    for x, y in zip(a, c):
        assert np.array_equal(x, y)


def test_gated_oracle_rejects_bad_arguments():
    rng = np.random.default_rng(24)
    q, k, v, b, cu, S0 = _problem(rng, 6, 2, 4, 3)
    with pytest.raises(ValueError):
        kda_recurrent_gated(q, k, v, np.zeros_like(q), np.zeros(3), b, cu)  # A_log must be [H]
    with pytest.raises(RuntimeError):
        kda_recurrent_gated(q, k, v, np.zeros_like(q), np.zeros(2), b, cu, mutation=3)  # not a gate mutation


# --- the unbounded form g = -e^{A_h} Softplus(z) (the mapping table's other row) ---------------

from oracle import UNBOUNDED_MUTATIONS, kda_recurrent_unbounded  # noqa: E402

NO_BOUND = -1.0e300  # a clamp no finite log-decay reaches


def _unbounded(mutation):
    def run(q, k, v, z, A, b, cu, S0):
        return kda_recurrent_unbounded(q, k, v, z, A, b, cu, init_state=S0, num_threads=2, mutation=mutation)
    return run


def _plain(q, k, v, g, b, cu, S0):
    return kda_recurrent(q, k, v, g, b, cu, lower_bound=NO_BOUND, init_state=S0, num_threads=2)


def pin_unbounded_closed_forms(run):
    """Softplus(0) = ln 2, Softplus(ln(e - 1)) = 1, Softplus(ln 3) = 2 ln 2: g = -e^{A_h} times these,
    per head; with A_h = ln 3 and z = ln 3 the decay is 6 ln 2 (alpha = 1/64), far below -5."""
    rng = np.random.default_rng(30)
    q, k, v, b, cu, S0 = _problem(rng, 17, 3, 6, 5)
    zs = np.array([0.0, np.log(np.e - 1.0), np.log(3.0)])
    A = np.array([0.0, -1.0, np.log(3.0)])
    z = np.broadcast_to(zs[rng.integers(0, 3, size=q.shape)], q.shape).copy()
    sp = np.where(z == 0.0, np.log(2.0), np.where(z == np.log(3.0), 2.0 * np.log(2.0), 1.0))
    g = -np.exp(A)[None, :, None] * sp
    _close(run(q, k, v, z, A, b, cu, S0), _plain(q, k, v, g, b, cu, S0), 1e-14)


def pin_unbounded_limits(run):
    """z -> -inf gives g = 0 (alpha = 1); for large z, Softplus(z) = z to fp64 precision, so
    g = -e^{A_h} z: at z = 40, A_h = 0 that is alpha = e^-40, a decay no bound of -5 allows."""
    rng = np.random.default_rng(31)
    q, k, v, b, cu, S0 = _problem(rng, 13, 2, 5, 4)
    z = np.where(rng.standard_normal(q.shape) > 0, -800.0, 40.0)
    A = np.array([0.0, 0.0])
    g = np.where(z < 0, 0.0, -40.0)
    _close(run(q, k, v, z, A, b, cu, S0), _plain(q, k, v, g, b, cu, S0), 1e-13)


UNBOUNDED_PINS = [pin_unbounded_closed_forms, pin_unbounded_limits]


@pytest.mark.parametrize("pin", UNBOUNDED_PINS, ids=lambda p: p.__name__)
def test_unbounded_pins(pin):
    pin(_unbounded(0))


@pytest.mark.parametrize("name", sorted(UNBOUNDED_MUTATIONS))
def test_planted_unbounded_mistake_is_caught(name):
    failed = []
    for pin in UNBOUNDED_PINS:
        try:
            pin(_unbounded(UNBOUNDED_MUTATIONS[name]))
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught {name}"


@pytest.mark.parametrize("chunk", [16, 32, 64])
def test_unbounded_chunked_form_agrees_with_recurrence(chunk):
    """The chunkwise form (oracle/chunked.py, every e^{G_t - G_i} formed from the difference,
    i.e. from position pairs) and the token recurrence agree for the unbounded map with steps
    of -80 on every third channel (far past the e^80 that a single reference could carry)
    and ordinary steps elsewhere, over packed sequences of lengths that are no multiple of the
    chunk."""
    from oracle.chunked import kda_chunked
    rng = np.random.default_rng(77)
    lens = [45, 1, 70]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, H, d = cu[-1], 2, 8
    q = rng.standard_normal((T, H, d))
    k = rng.standard_normal((T, H, d))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, d))
    z = -1.0 + 2.0 * rng.standard_normal((T, H, d))
    z[:, :, ::3] = 40.0
    A_log = np.array([np.log(2.0), -0.3])
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    init = 0.1 * rng.standard_normal((len(lens), H, d, d))
    g = -np.exp(A_log)[None, :, None] * (np.maximum(z, 0.0) + np.log1p(np.exp(-np.abs(z))))
    o_c, f_c = kda_chunked(q, k, v, g, beta, cu, chunk=chunk, lower_bound=-np.inf, init_state=init)
    o_r, f_r = kda_recurrent_unbounded(q, k, v, z, A_log, beta, cu, init_state=init, num_threads=2)
    scale_o, scale_f = np.sqrt(np.mean(o_r ** 2)), np.sqrt(np.mean(f_r ** 2))
    assert np.max(np.abs(o_c - o_r)) <= 1e-12 * scale_o and np.max(np.abs(f_c - f_r)) <= 1e-12 * scale_f
    assert g.min() < -70.0  # the steep steps are there
