"""CPU pins, in numpy fp64, of how the chunked kernel splits the decayed Gram entries of one
32-token chunk (Kimi K3 -- Architecture Notes, section 1.2, and the Kimi Linear treatment of
the diagonal tiles), against their definition

    A[t, i] = sum_c k_tc k_ic e^{G_tc - G_ic}  (i < t),    P[t, i] = sum_c q_tc k_ic e^{G_tc - G_ic}  (i <= t),

with G the cumulative log-decay inside the chunk. The kernel uses one reference r = G at the end
of the first 16-token subtile: f = e^{G - r} on the row side, g = e^{r - G} on the column side.
A channel whose log2-decay over a diagonal 16-token block is below -114 is "wide" there. Its
row factors (block 0: rows t < 16) or column factors (block 1: columns i >= 16) are left out of
the factored product, and its share of that block's entries comes from position pairs, one
exponential of a difference each. These tests check that the split reproduces the definition.
They also check that every factor the product keeps stays within the stated envelope: e^{+-80}
for decays >= -5 per token, 2^114 for the narrow channels of an unbounded map. A split with a
share left out, or with the reference moved, fails one of them."""

import numpy as np
import pytest

C, HALF, D = 32, 16, 24
WIDE = 114.0  # log2 units


def _chunk(rng, log_decay):
    q = rng.standard_normal((C, D))
    k = rng.standard_normal((C, D))
    G = np.cumsum(log_decay, axis=0)  # G[t, c]: log-decay of tokens 0..t (nats)
    return q, k, G


def _exact(x, k, G, strict):
    out = np.zeros((C, C))
    for t in range(C):
        for i in range(t if strict else t + 1):
            out[t, i] = np.sum(x[t] * k[i] * np.exp(G[t] - G[i]))
    return out


def _split(x, k, G, strict, *, ref=HALF - 1, drop_pairs=False, unbounded=True):
    """The kernel's form: factored product over the channels each entry keeps, plus position
    pairs for the channels wide in the entry's diagonal block (the unbounded map; the bounded
    maps keep every channel in the product). Returns (entries, largest log2 factor used)."""
    r = G[ref]
    G2 = G / np.log(2.0)
    wide0 = G2[HALF - 1] < -WIDE                  # block 0: tokens 0..15 (sum from the chunk start)
    wide1 = (G2[C - 1] - G2[HALF - 1]) < -WIDE    # block 1: tokens 16..31
    if not unbounded:
        wide0 = wide1 = np.zeros(D, bool)
    f = np.exp(G - r)
    g = np.exp(r - G)
    row_keep = np.ones((C, D), bool)
    row_keep[:HALF] &= ~wide0                     # rows t < 16 of the row-side operand
    col_keep = np.ones((C, D), bool)
    col_keep[HALF:] &= ~wide1                     # columns i >= 16 of the column-side operand
    out = np.zeros((C, C))
    used = -np.inf
    for t in range(C):
        for i in range(t if strict else t + 1):
            keep = row_keep[t] & col_keep[i]
            out[t, i] = np.sum((x[t] * f[t] * k[i] * g[i])[keep])
            if keep.any():
                used = max(used, np.log2(f[t][keep]).max(), np.log2(g[i][keep]).max())
            same_block = (t < HALF) == (i < HALF)
            if same_block and not drop_pairs:
                w = wide0 if t < HALF else wide1
                out[t, i] += np.sum((x[t] * k[i] * np.exp(G[t] - G[i]))[w])
    return out, used


def _close(a, b):
    return np.max(np.abs(a - b)) <= 1e-12 * max(1.0, np.max(np.abs(b)))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_bounded_decay_stays_inside_e80(seed):
    rng = np.random.default_rng(seed)
    la = -5.0 * rng.random((C, D))
    la[:, 0] = -5.0  # a channel at the bound on every token (e^80 = 2^115.4: still in fp32 range)
    q, k, G = _chunk(rng, la)
    for x, strict in ((k, True), (q, False)):
        got, used = _split(x, k, G, strict, unbounded=False)
        assert _close(got, _exact(x, k, G, strict))
        assert used <= 80.0 / np.log(2.0) + 1e-9  # e^80: 16 steps of -5 on either side of r


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_unbounded_decay_with_wide_channels(seed):
    rng = np.random.default_rng(10 + seed)
    la = -np.log1p(np.exp(2.0 * rng.standard_normal((C, D))))  # -Softplus(z), z ~ N(0, 4)
    la[:HALF, 1] = -12.0   # wide in block 0 only
    la[HALF:, 2] = -12.0   # wide in block 1 only
    la[:, 3] = -30.0       # wide in both
    la[:, 4] = -40.0 * rng.random(C)
    q, k, G = _chunk(rng, la)
    for x, strict in ((k, True), (q, False)):
        exact = _exact(x, k, G, strict)
        got, used = _split(x, k, G, strict)
        assert _close(got, exact)
        assert used <= WIDE + 1e-9  # the factors the tensor cores see
        # the same entries without the position pairs are wrong: the pairs carry the wide channels
        bad, _ = _split(x, k, G, strict, drop_pairs=True)
        assert not _close(bad, exact)


def test_moved_reference_leaves_the_envelope():
    # -4 per token keeps every channel narrow (64 nats, 92.3 in log2, per block); with r at the
    # chunk's last token the row factor of token 0 is e^{124}: past both e^80 and 2^114
    rng = np.random.default_rng(5)
    la = np.full((C, D), -4.0)
    q, k, G = _chunk(rng, la)
    for unbounded in (False, True):
        _, used = _split(k, k, G, True, unbounded=unbounded)
        assert used <= 80.0 / np.log(2.0)
        _, used = _split(k, k, G, True, ref=C - 1, unbounded=unbounded)
        assert used > WIDE


def test_every_channel_narrow_needs_no_pairs():
    rng = np.random.default_rng(7)
    la = -0.5 * rng.random((C, D))
    q, k, G = _chunk(rng, la)
    got, used = _split(q, k, G, False, drop_pairs=True)
    assert _close(got, _exact(q, k, G, False)) and used <= 16 * 0.5 / np.log(2.0) + 1e-9


def _back_substitution_row(A, j):
    """Row j of T = (I + A)^{-1} for strictly lower triangular A, as the inverse pair forms it:
    x^T (I + A) = e_j^T, i.e. x_m = [m == j] - sum_{i > m} x_i A[i][m], from m = n - 1 down."""
    n = A.shape[0]
    x = np.zeros(n)
    for m in range(n - 1, -1, -1):
        x[m] = (1.0 if m == j else 0.0) - sum(x[i] * A[i, m] for i in range(m + 1, n))
    return x


@pytest.mark.parametrize("seed", [0, 1])
def test_inverse_pair_back_substitution(seed):
    rng = np.random.default_rng(20 + seed)
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(C)))
    k = rng.standard_normal((C, D)); k /= np.linalg.norm(k, axis=1, keepdims=True)
    G = np.cumsum(-rng.uniform(0.0, 1.0, (C, D)), axis=0)
    A = np.zeros((C, C))  # A[t, i] = beta_t sum_c k_tc k_ic e^{G_tc - G_ic}, i < t
    for t in range(C):
        for i in range(t):
            A[t, i] = beta[t] * np.sum(k[t] * k[i] * np.exp(G[t] - G[i]))
    T = np.stack([_back_substitution_row(A, j) for j in range(C)])
    assert _close(T, np.linalg.inv(np.eye(C) + A))
    assert np.allclose(np.triu(T, 1), 0.0) and np.allclose(np.diag(T), 1.0)  # unit lower triangular
    # the same substitution with A transposed (A[m][i] where A[i][m] belongs) is not the inverse:
    # checked on the last row, which is dense
    j = C - 1
    x = np.zeros(C)
    for m in range(C - 1, -1, -1):
        x[m] = (1.0 if m == j else 0.0) - sum(x[i] * A[m, i] for i in range(m + 1, C))
    assert not _close(x, np.linalg.inv(np.eye(C) + A)[j])
