"""CPU pins, with the fp64 oracle, of the identity the segmented schedule for one long sequence
rests on. The recurrence S_t = (I - b_t k_t k_t^T) Diag(a_t) S_{t-1} + b_t k_t v_t^T (Kimi K3 --
Architecture Notes, section 1.1) is affine in the state. So a segment of tokens maps its
entering state S to M S + B, where B is the state the segment leaves from the zero state and M is
the state it leaves from the identity with v = 0. Chaining the segments' maps from the initial
state must give one full run's final state, and running each segment from its chained entering
state must give the full run's outputs for that segment. Cutting a segment at the wrong token,
or taking M with v left in, breaks them."""

import numpy as np
import pytest

from oracle import kda_recurrent

DK = DV = 6
H = 2


def _problem(rng, T, max_decay=0.3, beta_scale=1.0):
    """Mild decays keep M of order one over a segment, so that the entering state still matters."""
    q = rng.standard_normal((T, H, DK)); q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((T, H, DK)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, DV))
    la = -rng.uniform(0.0, max_decay, (T, H, DK))
    b = beta_scale / (1.0 + np.exp(-rng.standard_normal((T, H))))
    S0 = rng.standard_normal((1, H, DK, DV))
    return q, k, v, la, b, S0


def _run(q, k, v, la, b, a, e, init):
    return kda_recurrent(q[a:e], k[a:e], v[a:e], la[a:e], b[a:e], [0, e - a], init_state=init)


def _maps(q, k, v, la, b, a, e, *, v_in_m=False):
    """(M [H, dk, dk], B [H, dk, dv]) of tokens [a, e)."""
    _, B = _run(q, k, v, la, b, a, e, np.zeros((1, H, DK, DV)))
    eye = np.broadcast_to(np.eye(DK), (1, H, DK, DK)).copy()
    vm = v if v_in_m else np.zeros_like(q)  # width dk: the map acts on every column alike
    _, M = _run(q, k, vm, la, b, a, e, eye)
    return M[0], B[0]


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(1e-300, np.max(np.abs(b)))


@pytest.mark.parametrize("cuts", [[0, 13, 30, 45], [0, 1, 44, 45], [0, 15, 16, 17, 45]])
def test_chained_segment_maps_give_the_full_run(cuts):
    rng = np.random.default_rng(len(cuts) + cuts[1])
    T = cuts[-1]
    q, k, v, la, b, S0 = _problem(rng, T)
    out_full, S_full = kda_recurrent(q, k, v, la, b, [0, T], init_state=S0)
    S = S0[0]
    for a, e in zip(cuts[:-1], cuts[1:]):
        out_seg, S_seg = _run(q, k, v, la, b, a, e, S[None])
        assert _rel(out_seg, out_full[a:e]) < 1e-12  # the segment's outputs from its entering state
        M, B = _maps(q, k, v, la, b, a, e)
        S_next = np.einsum("hij,hjk->hik", M, S) + B
        assert _rel(S_next, S_seg[0]) < 1e-12  # the affine map is the segment's state update
        S = S_next
    assert _rel(S, S_full[0]) < 1e-12


def test_map_taken_with_v_is_wrong():
    rng = np.random.default_rng(3)
    q, k, v, la, b, S0 = _problem(rng, 30, max_decay=0.05, beta_scale=0.2)
    _, fin10 = _run(q, k, v, la, b, 0, 10, S0)
    M, B = _maps(q, k, v, la, b, 10, 30, v_in_m=True)  # (d_v = d_k here, so v fits the map's width)
    S_next = np.einsum("hij,hjk->hik", M, fin10[0]) + B
    assert _rel(S_next, _run(q, k, v, la, b, 10, 30, fin10)[1][0]) > 1e-3


def test_segment_cut_one_token_off_is_wrong():
    rng = np.random.default_rng(4)
    q, k, v, la, b, S0 = _problem(rng, 30, max_decay=0.05, beta_scale=0.2)
    _, fin12 = _run(q, k, v, la, b, 0, 12, S0)
    M, B = _maps(q, k, v, la, b, 13, 30)  # the map of [13, 30) applied at token 12
    _, S_true = _run(q, k, v, la, b, 12, 30, fin12)
    assert _rel(np.einsum("hij,hjk->hik", M, fin12[0]) + B, S_true[0]) > 1e-3
