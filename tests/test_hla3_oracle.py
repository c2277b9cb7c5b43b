"""Pins of the third-order oracle (``oracle/hla3_oracle.py``): closed forms, three algorithms
(triple sum, masked matrix products, streaming Y-form), the composition with the masked
second-order oracle, causality, and planted mistakes."""
import numpy as np
import pytest

from oracle import hla2_oracle as O2
from oracle import hla3_oracle as O3


def rnd(B, H, n, d, dv, seed=0, positive=False):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, H, n, d)) / np.sqrt(d)
    k = r.standard_normal((B, H, n, d)) / np.sqrt(d)
    v = r.standard_normal((B, H, n, dv))
    if positive:
        q, k = np.abs(q) + 0.1, np.abs(k) + 0.1
    return q, k, v


def rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


def test_closed_forms_n1_n2():
    q, k, v = rnd(1, 1, 2, 3, 2, seed=1)
    Q, K, V = q[0, 0], k[0, 0], v[0, 0]
    o = O3.serial_forward(q, k, v)[0, 0]
    assert np.allclose(o[0], (Q[0] @ K[0]) ** 3 * V[0], rtol=1e-13, atol=0)
    a = lambda t, s: Q[t] @ K[s]  # noqa: E731
    o2 = a(1, 0) * a(0, 0) * a(0, 0) * V[0]           # j = 1: i = l = 1
    for i in range(2):                                  # j = 2: i, l in {1, 2}
        for l in range(2):
            o2 = o2 + a(1, i) * a(1, i) * a(1, l) * V[l]
    assert np.allclose(o[1], o2, rtol=1e-12, atol=0)
    # the terms with i or l after j (excluded by the mask) are not negligible here
    full = sum(a(1, i) * a(j, i) * a(j, l) * V[l] for j in range(2) for i in range(2) for l in range(2))
    assert rel(full, o2) > 1e-3


@pytest.mark.parametrize("normalize", [False, True])
def test_three_algorithms_agree(normalize):
    q, k, v = rnd(2, 2, 8, 3, 2, seed=2, positive=normalize)
    a = O3.brute_force_forward(q, k, v, normalize)
    assert rel(O3.matrix_form_forward(q, k, v, normalize), a) < 1e-12
    assert rel(O3.serial_forward(q, k, v, normalize), a) < 1e-12


def test_composition_with_the_second_order_oracle():
    """Reading T4: the masked second-order output (the HLA-2 oracle, no decay) with the values
    replaced by the first-order outputs u_t = sum_{l <= t} (q_t . k_l) v_l."""
    q, k, v = rnd(1, 3, 21, 4, 3, seed=3)
    u = O3.first_order_forward(q, k, v)
    # the first-order form itself against its definition
    A = np.einsum("bhta,bhsa->bhts", q, k) * np.tril(np.ones((21, 21)))
    assert rel(u, A @ v) < 1e-12
    assert rel(O2.serial_forward(q, k, u), O3.serial_forward(q, k, v)) < 1e-12


def test_causality():
    q, k, v = rnd(1, 1, 12, 3, 2, seed=5)
    base = O3.serial_forward(q, k, v)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[..., 8:, :] += 1.0
    k2[..., 8:, :] -= 0.7
    v2[..., 8:, :] *= 2.0
    assert np.array_equal(O3.serial_forward(q2, k2, v2)[..., :8, :], base[..., :8, :])


def test_planted_mistakes_are_caught():
    """Dropping the l <= j mask (l <= t instead), or the partial-product mask (j free), or
    using P before the token's own update, breaks agreement with the triple sum."""
    q, k, v = rnd(1, 1, 7, 3, 2, seed=6)
    ref = O3.brute_force_forward(q, k, v)
    Q, K, V = q[0, 0], k[0, 0], v[0, 0]
    n = 7
    A = Q @ K.T
    M = np.tril(np.ones((n, n)))
    Am = A * M
    no_l_mask = ((Am @ Am.T) * M) @ (A * M[-1][None, :]) @ V      # l up to n, not j
    assert rel(no_l_mask, ref[0, 0]) > 1e-3
    no_j_mask = (Am @ Am.T) @ Am @ V                              # j unrestricted
    assert rel(no_j_mask, ref[0, 0]) > 1e-3
    # P read before its update at t
    S = np.zeros((3, 3))
    P = np.zeros((3, 2))
    Y = np.zeros((3, 2))
    bad = np.zeros((n, 2))
    for t in range(n):
        S = S + np.outer(K[t], K[t])
        u = Q[t] @ P
        P = P + np.outer(K[t], V[t])
        Y = Y + np.outer(S @ Q[t], u)
        bad[t] = Q[t] @ Y
    assert rel(bad, ref[0, 0]) > 1e-3


@pytest.mark.parametrize("normalize", [False, True])
def test_decode_from_zero_equals_the_triple_sum(normalize):
    """Streaming with the packed state [S^K | P^KV | Y | m^K | y] from zero reproduces the
    triple sum token by token (the masked streaming of the technical summary, item 3)."""
    q, k, v = rnd(2, 2, 9, 3, 2, seed=9, positive=normalize)
    ref = O3.brute_force_forward(q, k, v, normalize)
    state = np.zeros((2, 2, O3.state_floats(3, 2)))
    outs = [O3.decode_step(state, q[:, :, t], k[:, :, t], v[:, :, t], normalize) for t in range(9)]
    assert rel(np.stack(outs, axis=2), ref) < 1e-12
