"""Pins of the float64 oracle against facts fixed by the pages and by mathematics.

Nothing here compares the oracle with itself by retyping a formula: each pin is a
closed form, an exact rational evaluation, a different algorithm (pair sum vs serial
recurrence vs chunked scan vs matrix form), an invariant, or finite differences.
A final group plants plausible mistakes in copies of the oracle and checks that the
pins catch every one of them.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import cref
from oracle import hla2_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(B, H, n, d, dv, seed=0, positive=False):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, H, n, d)) / np.sqrt(d)
    k = r.standard_normal((B, H, n, d)) / np.sqrt(d)
    v = r.standard_normal((B, H, n, dv))
    if positive:
        q, k = np.log1p(np.exp(q * np.sqrt(d))), np.log1p(np.exp(k * np.sqrt(d)))
    return q, k, v


def rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


# ---------------------------------------------------------------------------
# Closed forms and exact values
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("g", [1.0, 0.7])
def test_single_token_closed_form(g):
    """n = 1: o_1 = (q_1 . k_1)^2 v_1 whatever the decay."""
    q, k, v = rnd(1, 1, 1, 5, 3, seed=1)
    o = O.serial_forward(q, k, v, [g])
    expect = (q[0, 0, 0] @ k[0, 0, 0]) ** 2 * v[0, 0, 0]
    np.testing.assert_allclose(o[0, 0, 0], expect, rtol=1e-13)


@pytest.mark.parametrize("g", [1.0, 0.6])
def test_two_token_closed_form(g):
    """n = 2: o_2 = g^2 (q2.k1)(k1.q1) v1 + g (q2.k1)^2 v2 + (q2.k2)^2 v2.
    The pair (key 2, value 1) is absent: that is the mask."""
    q, k, v = rnd(1, 1, 2, 4, 3, seed=2)
    q1, q2 = q[0, 0]
    k1, k2 = k[0, 0]
    v1, v2 = v[0, 0]
    expect = g * g * (q2 @ k1) * (k1 @ q1) * v1 + g * (q2 @ k1) ** 2 * v2 + (q2 @ k2) ** 2 * v2
    o = O.serial_forward(q, k, v, [g])
    np.testing.assert_allclose(o[0, 0, 1], expect, rtol=1e-12)
    leaked = g * (q2 @ k2) * (k2 @ q1) * v1
    assert np.max(np.abs(leaked)) > 1e-3  # the excluded pair is not negligible here


def test_scalar_feature_closed_form():
    """d = 1: o_t = q_t * sum_{i<=j<=t} g^((t-i)+(t-j)) k_i^2 q_j v_j."""
    q, k, v = rnd(1, 1, 7, 1, 2, seed=3)
    g = 0.8
    o = O.serial_forward(q, k, v, [g])
    Q, K, V = q[0, 0, :, 0], k[0, 0, :, 0], v[0, 0]
    for t in range(7):
        s = sum(g ** ((t - i) + (t - j)) * K[i] ** 2 * Q[j] * V[j]
                for j in range(t + 1) for i in range(j + 1))
        np.testing.assert_allclose(o[0, 0, t], Q[t] * s, rtol=1e-12)


@pytest.mark.parametrize("name", ["n2_d1", "n5_d2", "n4_d3_nodecay"])
@pytest.mark.parametrize("impl", ["numpy", "c"])
def test_exact_rational_fixtures(name, impl):
    """Serial float64 recurrence against exact rational pair sums (tests/golden)."""
    with open(os.path.join(GOLDEN, f"{name}.json")) as f:
        doc = json.load(f)
    q = np.array(doc["q"], dtype=np.float64)[None, None]
    k = np.array(doc["k"], dtype=np.float64)[None, None]
    v = np.array(doc["v"], dtype=np.float64)[None, None]
    g = float(Fraction(doc["gamma"]))
    out = np.array([[float(Fraction(x)) for x in row] for row in doc["out"]])
    den = np.array([float(Fraction(x)) for x in doc["den"]])
    if impl == "numpy":
        o = O.serial_forward(q, k, v, [g])[0, 0]
        on = O.serial_forward(q, k, v, [g], normalize=True, eps=0.0)[0, 0]
    else:
        o = cref.forward(q, k, v, [g])[0, 0]
        on = cref.forward(q, k, v, [g], normalize=True, eps=0.0)[0, 0]
    np.testing.assert_allclose(o, out, rtol=1e-13, atol=1e-12)
    np.testing.assert_allclose(on, out / den[:, None], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# Three algorithms, one function
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("g", [None, 0.9])
@pytest.mark.parametrize("normalize", [False, True])
def test_brute_force_equals_serial(g, normalize):
    q, k, v = rnd(2, 2, 9, 3, 2, seed=4, positive=normalize)
    gam = None if g is None else [g, g * 0.95]
    a = O.brute_force_forward(q, k, v, gam, normalize=normalize)
    b = O.serial_forward(q, k, v, gam, normalize=normalize)
    assert rel(b, a) < 1e-12


def test_matrix_form_equals_serial():
    """Matrix form (A A^T V structure of the technical summary, item 2, with masks):
    with A = Q K^T and Atil = lower-triangular part of A (i <= j),
        W = ((A * Gam) Atil^T) * Gam_low,   O = W V,
    where Gam[t, i] = g^(t-i) and Gam_low[t, j] = g^(t-j) [j <= t]."""
    q, k, v = rnd(1, 1, 23, 5, 4, seed=5)
    g = 0.93
    Q, K, V = q[0, 0], k[0, 0], v[0, 0]
    n = Q.shape[0]
    A = Q @ K.T
    idx = np.arange(n)
    lag = idx[:, None] - idx[None, :]
    Gam = g ** lag.astype(np.float64)
    Atil = np.tril(A)
    W = ((A * np.where(lag >= 0, Gam, 0.0)) @ Atil.T) * np.where(lag >= 0, Gam, 0.0)
    o = O.serial_forward(q, k, v, [g])[0, 0]
    assert rel(o, W @ V) < 1e-12


@pytest.mark.parametrize("chunk", [1, 2, 3, 4, 5, 16, 13])
def test_chunked_scan_equals_serial_any_width(chunk):
    """Chunk-width independence ([PS] §4, [TS4]): the scan reproduces the serial
    recurrence for every chunk width, including non-divisors of n."""
    q, k, v = rnd(1, 2, 13, 3, 2, seed=6)
    gam = [0.85, 1.0]
    a, sa = O.serial_forward(q, k, v, gam, return_state=True)
    b, sb = O.chunked_scan_forward(q, k, v, gam, chunk=chunk, return_state=True)
    assert rel(b, a) < 1e-12
    for key in ("S", "C", "m", "G", "h"):
        assert rel(sb[key], sa[key]) < 1e-12


def test_chunked_scan_normalized_and_init_state():
    q, k, v = rnd(1, 1, 10, 3, 2, seed=7, positive=True)
    q0, k0, v0 = rnd(1, 1, 6, 3, 2, seed=8, positive=True)
    _, init = O.serial_forward(q0, k0, v0, [0.9], return_state=True)
    a = O.serial_forward(q, k, v, [0.9], normalize=True, init_state=init)
    b = O.chunked_scan_forward(q, k, v, [0.9], chunk=4, normalize=True, init_state=init)
    assert rel(b, a) < 1e-12


# ---------------------------------------------------------------------------
# Algebra of the combine
# ---------------------------------------------------------------------------

def _rand_tuple(r, d, dv):
    return {"S": r.standard_normal((d, d)), "C": r.standard_normal((d, dv)),
            "m": r.standard_normal(d), "G": r.standard_normal((d, dv)),
            "h": r.standard_normal(d), "rho": float(r.uniform(0.2, 1.0))}


def test_combine_associative():
    r = np.random.default_rng(9)
    for _ in range(20):
        a, b, c = (_rand_tuple(r, 4, 3) for _ in range(3))
        x = O.combine(O.combine(a, b), c)
        y = O.combine(a, O.combine(b, c))
        for key in ("S", "C", "m", "G", "h"):
            assert rel(x[key], y[key]) < 1e-13
        assert abs(x["rho"] - y["rho"]) < 1e-15


def test_combine_identity():
    r = np.random.default_rng(10)
    a = _rand_tuple(r, 3, 2)
    e = O.identity_element(3, 2)
    for x in (O.combine(a, e), O.combine(e, a)):
        for key in ("S", "C", "m", "G", "h"):
            np.testing.assert_array_equal(x[key], a[key])


def test_combine_not_commutative():
    """Time order matters: swapping segments changes the masked summaries."""
    r = np.random.default_rng(11)
    a, b = _rand_tuple(r, 3, 2), _rand_tuple(r, 3, 2)
    assert rel(O.combine(a, b)["G"], O.combine(b, a)["G"]) > 1e-3


def test_blelloch_matches_sequential_fold():
    r = np.random.default_rng(12)
    items = [_rand_tuple(r, 3, 2) for _ in range(11)]
    pre = O.blelloch_exclusive_scan(items, 3, 2)
    acc = O.identity_element(3, 2)
    for i, it in enumerate(items):
        for key in ("S", "C", "m", "G", "h"):
            np.testing.assert_allclose(pre[i][key], acc[key], rtol=1e-12, atol=1e-12)
        acc = O.combine(acc, it)


# ---------------------------------------------------------------------------
# Invariants
# ---------------------------------------------------------------------------

def test_gamma_one_equals_no_decay():
    q, k, v = rnd(1, 3, 8, 3, 2, seed=13)
    a = O.serial_forward(q, k, v, None)
    b = O.serial_forward(q, k, v, [1.0, 1.0, 1.0])
    np.testing.assert_array_equal(a, b)
    # and as g -> 1 the decayed output converges to it
    c = O.serial_forward(q, k, v, [1 - 1e-9] * 3)
    assert rel(c, a) < 1e-7


def test_z_form_identity():
    """q^T (S_t C_t - G_t) = q^T Z_t with Z_t = g^2 Z_{t-1} + S_t q_t v_t^T; and the
    denominator S_t m_t - h_t = y_t with y_t = g^2 y_{t-1} + S_t q_t."""
    q, k, v = rnd(1, 1, 17, 4, 3, seed=14, positive=True)
    g = 0.91
    o, st = O.serial_forward(q, k, v, [g], return_state=True)
    Q, K, V = q[0, 0], k[0, 0], v[0, 0]
    S = np.zeros((4, 4))
    Z = np.zeros((4, 3))
    y = np.zeros(4)
    for t in range(17):
        S = g * S + np.outer(K[t], K[t])
        p = S @ Q[t]
        Z = g * g * Z + np.outer(p, V[t])
        y = g * g * y + p
        np.testing.assert_allclose(Q[t] @ Z, o[0, 0, t], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(Z, st["S"][0, 0] @ st["C"][0, 0] - st["G"][0, 0], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(y, st["S"][0, 0] @ st["m"][0, 0] - st["h"][0, 0], rtol=1e-11, atol=1e-13)


def test_causality():
    q, k, v = rnd(1, 1, 12, 3, 2, seed=15)
    o = O.serial_forward(q, k, v, [0.9])
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    r = np.random.default_rng(16)
    q2[..., 7:, :] += r.standard_normal(q2[..., 7:, :].shape)
    k2[..., 7:, :] += r.standard_normal(k2[..., 7:, :].shape)
    v2[..., 7:, :] += r.standard_normal(v2[..., 7:, :].shape)
    o2 = O.serial_forward(q2, k2, v2, [0.9])
    np.testing.assert_array_equal(o[..., :7, :], o2[..., :7, :])
    assert rel(o2[..., 7:, :], o[..., 7:, :]) > 1e-3


def test_masked_vs_unmasked_difference_is_G():
    """q^T S_t C_t - o_t = q^T G_t, and G_t equals the pair sum over key index > value index."""
    q, k, v = rnd(1, 1, 6, 3, 2, seed=17)
    g = 0.8
    o, st = O.serial_forward(q, k, v, [g], return_state=True)
    Q, K, V = q[0, 0], k[0, 0], v[0, 0]
    t = 5
    unmasked = Q[t] @ st["S"][0, 0] @ st["C"][0, 0]
    np.testing.assert_allclose(unmasked - o[0, 0, t], Q[t] @ st["G"][0, 0], rtol=1e-12)
    Gb = sum(g ** ((t - i) + (t - j)) * np.outer(K[i], K[i]) @ np.outer(Q[j], V[j])
             for i in range(t + 1) for j in range(i))
    np.testing.assert_allclose(st["G"][0, 0], Gb, rtol=1e-12)


def test_streaming_equals_forward_and_continuation():
    """Token-at-a-time decode from zero equals the forward; splitting the sequence
    and continuing from the first part's final state equals one pass."""
    q, k, v = rnd(2, 3, 14, 4, 3, seed=18)
    gam = [0.9, 0.97, 1.0]
    full, fst = O.serial_forward(q, k, v, gam, return_state=True)
    _, s1 = O.serial_forward(q[:, :, :9], k[:, :, :9], v[:, :, :9], gam, return_state=True)
    tail, s2 = O.serial_forward(q[:, :, 9:], k[:, :, 9:], v[:, :, 9:], gam, init_state=s1,
                                return_state=True)
    assert rel(tail, full[:, :, 9:]) < 1e-13
    for key in fst:
        assert rel(s2[key], fst[key]) < 1e-13
    # packed layout round trip
    np.testing.assert_array_equal(O.pack_state(O.unpack_state(O.pack_state(fst), 4, 3)),
                                  O.pack_state(fst))


# ---------------------------------------------------------------------------
# Gradients ([PS] §4.2 reverse mode)
# ---------------------------------------------------------------------------

def _loss(q, k, v, dO, g):
    return float(np.sum(O.serial_forward(q, k, v, g) * dO))


def test_adjoint_matches_finite_differences():
    q, k, v = rnd(1, 1, 7, 3, 2, seed=19)
    dO = np.random.default_rng(20).standard_normal(v.shape)
    g = [0.88]
    dq, dk, dvv = O.serial_backward(q, k, v, dO, g)
    eps = 1e-6
    for arr, grad in ((q, dq), (k, dk), (v, dvv)):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            a0 = arr[idx]
            arr[idx] = a0 + eps
            lp = _loss(q, k, v, dO, g)
            arr[idx] = a0 - eps
            lm = _loss(q, k, v, dO, g)
            arr[idx] = a0
            num[idx] = (lp - lm) / (2 * eps)
        assert rel(grad, num) < 1e-7


def _fd_normalized(q, k, v, dO, g, eps, h=1e-6):
    """Central differences of L = sum dO . o_norm with respect to q, k, v."""
    def loss():
        return float(np.sum(O.serial_forward(q, k, v, g, normalize=True, eps=eps) * dO))

    out = []
    for arr in (q, k, v):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            a0 = arr[idx]
            arr[idx] = a0 + h
            lp = loss()
            arr[idx] = a0 - h
            lm = loss()
            arr[idx] = a0
            num[idx] = (lp - lm) / (2 * h)
        out.append(num)
    return out


def test_normalized_adjoint_matches_finite_differences():
    """The quotient-rule adjoint of the ratio-normalised output ([PS] §5.1, reading R4)
    against central differences of the normalised serial forward itself."""
    q, k, v = rnd(1, 1, 6, 3, 2, seed=31, positive=True)
    dO = np.random.default_rng(32).standard_normal(v.shape)
    g, eps = [0.9], 1e-3
    got = O.serial_backward_normalized(q, k, v, dO, g, eps)
    for a, b in zip(got, _fd_normalized(q, k, v, dO, g, eps)):
        assert rel(a, b) < 1e-6


def test_normalized_adjoint_c_matches_numpy():
    q, k, v = rnd(2, 2, 40, 4, 3, seed=33, positive=True)
    dO = np.random.default_rng(34).standard_normal(v.shape)
    g = [0.97, 0.999]
    # the C path sees float32 inputs: round them first so both sides use the same values
    q, k, v = (x.astype(np.float32).astype(np.float64) for x in (q, k, v))
    a = O.serial_backward_normalized(q, k, v, dO, g, 1e-6)
    b = cref.backward_normalized(q, k, v, dO, g, 1e-6)
    for x, y in zip(a, b):
        assert rel(x, y) < 1e-5


def test_planted_dropped_denominator_path_is_caught(monkeypatch):
    """Dropping the denominator's path of the quotient rule (a plausible mistake) makes the
    normalised adjoint disagree with finite differences."""
    q, k, v = rnd(1, 1, 5, 2, 2, seed=35, positive=True)
    dO = np.random.default_rng(36).standard_normal(v.shape)
    g, eps = [0.9], 1e-3
    fd = _fd_normalized(q, k, v, dO, g, eps)
    real = O.serial_backward

    def numerator_only(q_, k_, v_, d_, g_=None):
        if v_.shape[-1] == 1 and np.all(v_ == 1.0):
            z = np.zeros_like(np.asarray(q_, dtype=np.float64))
            return z, z.copy(), np.zeros_like(np.asarray(v_, dtype=np.float64))
        return real(q_, k_, v_, d_, g_)

    monkeypatch.setattr(O, "serial_backward", numerator_only)
    bad = O.serial_backward_normalized(q, k, v, dO, g, eps)
    assert rel(bad[0], fd[0]) > 1e-3 or rel(bad[1], fd[1]) > 1e-3


def test_adjoint_matches_pairsum_gradients():
    q, k, v = rnd(1, 2, 8, 3, 2, seed=21)
    dO = np.random.default_rng(22).standard_normal(v.shape)
    g = [0.9, 1.0]
    a = O.serial_backward(q, k, v, dO, g)
    b = O.pairsum_grads(q, k, v, dO, g)
    for x, y in zip(a, b):
        assert rel(x, y) < 1e-11


def test_adjoint_dot_test():
    """<dO, J dx> = <J^T dO, dx> for a random direction dx (linearisation by central
    differences of the forward)."""
    q, k, v = rnd(1, 1, 9, 3, 3, seed=23)
    r = np.random.default_rng(24)
    dO = r.standard_normal(v.shape)
    dq_, dk_, dv_ = (r.standard_normal(x.shape) for x in (q, k, v))
    g = [0.95]
    h = 1e-6
    fp = O.serial_forward(q + h * dq_, k + h * dk_, v + h * dv_, g)
    fm = O.serial_forward(q - h * dq_, k - h * dk_, v - h * dv_, g)
    lhs = np.sum(dO * (fp - fm) / (2 * h))
    gq, gk, gv = O.serial_backward(q, k, v, dO, g)
    rhs = np.sum(gq * dq_) + np.sum(gk * dk_) + np.sum(gv * dv_)
    assert abs(lhs - rhs) / abs(rhs) < 1e-7


# ---------------------------------------------------------------------------
# The C oracle agrees with the numpy oracle
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("masked", [True, False])
@pytest.mark.parametrize("normalize", [False, True])
def test_c_oracle_forward_matches_numpy(normalize, masked):
    q, k, v = rnd(2, 3, 40, 8, 5, seed=25, positive=normalize)
    q, k, v = (x.astype(np.float32).astype(np.float64) for x in (q, k, v))
    gam = [0.9, 0.99, 1.0]
    a, sa = O.serial_forward(q, k, v, gam, normalize=normalize, return_state=True, masked=masked)
    b, sb = cref.forward(q, k, v, gam, normalize=normalize, return_state=True, masked=masked)
    assert rel(b, a) < 1e-12
    assert rel(sb, O.pack_state(sa)) < 1e-12
    # continuation from a packed state
    c = cref.forward(q, k, v, gam, normalize=normalize, init_state=sb, masked=masked)
    d_ = O.serial_forward(q, k, v, gam, normalize=normalize, init_state=sa, masked=masked)
    assert rel(c, d_) < 1e-12


@pytest.mark.parametrize("masked", [True, False])
def test_c_oracle_decode_matches_numpy(masked):
    q, k, v = rnd(3, 2, 5, 6, 4, seed=26)
    q, k, v = (x.astype(np.float32).astype(np.float64) for x in (q, k, v))
    gam = [0.9, 0.999]
    st = np.zeros((3, 2, O.state_floats(6, 4)))
    outs = []
    for t in range(5):
        outs.append(cref.decode_step(st, q[:, :, t], k[:, :, t], v[:, :, t], gam, masked=masked))
    a = O.serial_forward(q, k, v, gam, masked=masked)
    assert rel(np.stack(outs, axis=2), a) < 1e-12


def test_c_oracle_backward_matches_numpy():
    q, k, v = rnd(1, 2, 37, 5, 4, seed=27)
    q, k, v = (x.astype(np.float32).astype(np.float64) for x in (q, k, v))
    dO = np.random.default_rng(28).standard_normal(v.shape).astype(np.float32).astype(np.float64)
    gam = [0.93, 1.0]
    a = O.serial_backward(q, k, v, dO, gam)
    b = cref.backward(q, k, v, dO, gam)
    for x, y in zip(a, b):
        assert rel(y, x) < 1e-11


# ---------------------------------------------------------------------------
# Planted mistakes: each plausible error in the recurrence breaks a pin
# ---------------------------------------------------------------------------

def _mutant_step(kind):
    def step(state, q_t, k_t, v_t, g, normalize=False, eps=1e-6, masked=True):
        gg = g[None, :]
        S, C, m, G, h = state["S"], state["C"], state["m"], state["G"], state["h"]
        gG = gg * gg if kind != "G_decay_once" else gg
        S1 = gg[..., None, None] * S + np.einsum("bha,bhc->bhac", k_t, k_t)
        C1 = gg[..., None, None] * C + np.einsum("bha,bhe->bhae", q_t, v_t)
        Csrc = C1 if kind == "G_uses_new_C" else C
        kC = np.einsum("bha,bhae->bhe", k_t, Csrc)
        sign = -1.0 if kind == "G_sign" else 1.0
        G1 = gG[..., None, None] * G + sign * gg[..., None, None] * np.einsum("bha,bhe->bhae", k_t, kC)
        if kind == "G_transposed_key":
            G1 = gG[..., None, None] * G + gg[..., None, None] * np.einsum("bha,bhe->bhae", q_t, kC)
        m1 = gg[..., None] * m + q_t
        u = np.einsum("bha,bhac->bhc", q_t, S1)
        o = np.einsum("bhc,bhce->bhe", u, C1) - np.einsum("bha,bhae->bhe", q_t, G1)
        return {"S": S1, "C": C1, "m": m1, "G": G1, "h": h}, o
    return step


@pytest.mark.parametrize("kind", ["G_uses_new_C", "G_decay_once", "G_sign", "G_transposed_key"])
def test_planted_mistakes_are_caught(kind, monkeypatch):
    q, k, v = rnd(1, 1, 6, 3, 2, seed=29)
    g = [0.8]
    truth = O.brute_force_forward(q, k, v, g)
    monkeypatch.setattr(O, "step", _mutant_step(kind))
    bad = O.serial_forward(q, k, v, g)
    assert rel(bad, truth) > 1e-3


def test_planted_combine_mistake_is_caught(monkeypatch):
    """Cross term on the wrong side (S_A C_B instead of S_B C_A) breaks chunk-width
    independence."""
    q, k, v = rnd(1, 1, 8, 3, 3, seed=30)
    truth = O.serial_forward(q, k, v, [0.9])
    orig = O.combine

    def wrong(A, B):
        out = orig(A, B)
        r = B["rho"]
        out["G"] = r * r * A["G"] + B["G"] + r * (A["S"] @ B["C"])
        return out

    monkeypatch.setattr(O, "combine", wrong)
    bad = O.chunked_scan_forward(q, k, v, [0.9], chunk=4)
    assert rel(bad, truth) > 1e-3


# ---------------------------------------------------------------------------
# Compact decode layout (S symmetric: upper block triangle only)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("d,dv", [(16, 16), (32, 64), (128, 128)])
def test_compact_layout_size_and_roundtrip(d, dv):
    """d (d + 4) / 2 floats for S (the upper triangle plus the lower halves of the 4 x 4
    diagonal blocks); a symmetric S survives the round trip exactly."""
    r = np.random.default_rng(d + dv)
    A = r.standard_normal((2, 3, d, d))
    S = A + np.swapaxes(A, -1, -2)
    rest = r.standard_normal((2, 3, 2 * d * dv + 2 * d))
    flat = np.concatenate([S.reshape(2, 3, d * d), rest], axis=-1)
    c = O.compact_from_state(flat, d, dv)
    assert c.shape[-1] == O.compact_state_floats(d, dv) == d * (d + 4) // 2 + 2 * d * dv + 2 * d
    assert np.array_equal(O.state_from_compact(c, d, dv), flat)
    # row 5 of S starts after rows 0..3 (d floats each) and row 4 (d - 4 floats)
    assert np.array_equal(c[..., 4 * d + (d - 4): 4 * d + (d - 4) + (d - 4)], S[..., 5, 4:])


def test_compact_state_continues_the_serial_recurrence():
    """A decode step on the expanded compact state equals one on the original state: the
    state's S is symmetric, so nothing is lost (serial recurrence of the pages)."""
    q, k, v = rnd(1, 2, 9, 8, 4, seed=41)
    _, st = O.serial_forward(q, k, v, [0.9, 0.99], return_state=True)
    flat = O.pack_state(st)
    back = O.unpack_state(O.state_from_compact(O.compact_from_state(flat, 8, 4), 8, 4), 8, 4)
    for key in ("S", "C", "G", "m", "h"):
        assert np.allclose(back[key], st[key], rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Unmasked variant (reading R6): o_t = q_t^T S_t C_t, the unmasked monoid
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("g", [1.0, 0.7])
def test_unmasked_closed_form_n2(g):
    """n = 2 written out: every (key, value) pair of S_2 C_2 is kept, including the pair
    (key 2, value 1) that the mask removes."""
    q, k, v = rnd(1, 1, 2, 3, 2, seed=40)
    Q, K, V = q[0, 0], k[0, 0], v[0, 0]
    o = O.serial_forward(q, k, v, [g], masked=False)[0, 0]
    assert np.allclose(o[0], (Q[0] @ K[0]) ** 2 * V[0], rtol=1e-13, atol=0)
    S2 = g * np.outer(K[0], K[0]) + np.outer(K[1], K[1])
    C2 = g * np.outer(Q[0], V[0]) + np.outer(Q[1], V[1])
    assert np.allclose(o[1], Q[1] @ S2 @ C2, rtol=1e-13, atol=0)
    masked = O.serial_forward(q, k, v, [g])[0, 0]
    removed = g * (Q[1] @ K[1]) * (K[1] @ Q[0]) * V[0]   # key index 2 > value index 1
    assert np.allclose(o[1] - masked[1], removed, rtol=1e-12, atol=1e-15)


def test_unmasked_last_row_is_a_at_v():
    """Without decay the last token sees the whole sequence, so its unmasked output is the
    last row of A A^T V with A = Q K^T (the symmetric structure of the technical summary),
    computed here with library matmuls."""
    q, k, v = rnd(2, 2, 9, 4, 3, seed=41)
    o = O.serial_forward(q, k, v, masked=False)
    for b in range(2):
        for h in range(2):
            A = q[b, h] @ k[b, h].T
            assert rel(o[b, h, -1], (A @ A.T @ v[b, h])[-1]) < 1e-12
            # and every row t is the same product restricted to the first t + 1 tokens
            t = 4
            At = q[b, h, :t + 1] @ k[b, h, :t + 1].T
            assert rel(o[b, h, t], (At @ At.T @ v[b, h, :t + 1])[-1]) < 1e-12


@pytest.mark.parametrize("normalize", [False, True])
def test_unmasked_brute_force_equals_serial(normalize):
    q, k, v = rnd(1, 2, 8, 3, 2, seed=42, positive=normalize)
    g = [1.0, 0.85]
    assert rel(O.serial_forward(q, k, v, g, normalize, masked=False),
               O.brute_force_forward(q, k, v, g, normalize, masked=False)) < 1e-12


@pytest.mark.parametrize("chunk", [1, 2, 3, 5, 16])
def test_unmasked_chunked_scan_equals_serial(chunk):
    q, k, v = rnd(2, 2, 13, 3, 2, seed=43)
    g = [0.9, 1.0]
    out, fin = O.chunked_scan_forward(q, k, v, g, chunk, masked=False, return_state=True)
    ref, st = O.serial_forward(q, k, v, g, masked=False, return_state=True)
    assert rel(out, ref) < 1e-12
    for key in ("S", "C", "m"):
        assert rel(fin[key], st[key]) < 1e-12
    assert not fin["G"].any() and not fin["h"].any()
    qp, kp, vp = rnd(1, 1, 10, 3, 2, seed=44, positive=True)
    assert rel(O.chunked_scan_forward(qp, kp, vp, [0.95], chunk, normalize=True, masked=False),
               O.serial_forward(qp, kp, vp, [0.95], normalize=True, masked=False)) < 1e-12


def test_unmasked_continuation_from_state():
    """The unmasked scan seeded with the serial state after t0 tokens continues exactly."""
    q, k, v = rnd(1, 2, 12, 3, 2, seed=45)
    g = [0.9, 0.97]
    full = O.serial_forward(q, k, v, g, masked=False)
    _, st = O.serial_forward(q[:, :, :5], k[:, :, :5], v[:, :, :5], g, masked=False, return_state=True)
    rest = O.chunked_scan_forward(q[:, :, 5:], k[:, :, 5:], v[:, :, 5:], g, 3, init_state=st, masked=False)
    assert rel(rest, full[:, :, 5:]) < 1e-12


def test_unmasked_monoid_algebra():
    """Associative with an identity; at g = 1 it is commutative (plain sums), which the
    masked semidirect product is not."""
    r = np.random.default_rng(46)

    def item(rho):
        return {"S": r.standard_normal((3, 3)), "C": r.standard_normal((3, 2)),
                "m": r.standard_normal(3), "rho": rho}

    X, Y, Z = item(0.9), item(0.6), item(0.8)
    left = O.combine_unmasked(O.combine_unmasked(X, Y), Z)
    right = O.combine_unmasked(X, O.combine_unmasked(Y, Z))
    for key in ("S", "C", "m"):
        assert rel(left[key], right[key]) < 1e-13
    e = O.unmasked_identity(3, 2)
    for key in ("S", "C", "m"):
        assert np.array_equal(O.combine_unmasked(e, X)[key], X[key])
        assert np.array_equal(O.combine_unmasked(X, e)[key], X[key])
    X1, Y1 = item(1.0), item(1.0)
    for key in ("S", "C", "m"):
        assert np.array_equal(O.combine_unmasked(X1, Y1)[key], O.combine_unmasked(Y1, X1)[key])


def test_unmasked_planted_mistakes_are_caught(monkeypatch):
    """A cross term in the unmasked monoid, or C decayed by g^2, breaks the agreement with
    the serial recurrence; so does dropping the diagonal-and-later pairs (the masked sum)."""
    q, k, v = rnd(1, 1, 9, 3, 2, seed=47)
    truth = O.serial_forward(q, k, v, [0.9], masked=False)
    assert rel(O.serial_forward(q, k, v, [0.9]), truth) > 1e-3
    orig = O.combine_unmasked

    def with_cross(A, B):
        out = orig(A, B)
        out["C"] = out["C"] + B["rho"] * (B["S"] @ A["C"])
        return out

    monkeypatch.setattr(O, "combine_unmasked", with_cross)
    assert rel(O.chunked_scan_forward(q, k, v, [0.9], 3, masked=False), truth) > 1e-3

    def c_decay_twice(A, B):
        out = orig(A, B)
        out["C"] = B["rho"] ** 2 * A["C"] + B["C"]
        return out

    monkeypatch.setattr(O, "combine_unmasked", c_decay_twice)
    assert rel(O.chunked_scan_forward(q, k, v, [0.9], 3, masked=False), truth) > 1e-3


# ---------------------------------------------------------------------------
# Multi-query sharing of S (reading R7)
# ---------------------------------------------------------------------------

def _mq_run(q, k, v, gam, group, normalize=False, masked=True, S_step=None):
    """Stream all tokens through the multi-query decode step from the empty state."""
    N, Hk, n, d = k.shape
    H, dv = Hk * group, v.shape[-1]
    S = np.zeros((N, Hk, d, d))
    heads = {"C": np.zeros((N, H, d, dv)), "G": np.zeros((N, H, d, dv)), "m": np.zeros((N, H, d)),
             "h": np.zeros((N, H, d))}
    step = S_step or O.mq_decode_step
    outs = []
    for t in range(n):
        S, heads, o = step(S, heads, q[:, :, t], k[:, :, t], v[:, :, t], gam, group, normalize, 1e-6, masked)
        outs.append(o)
    return np.stack(outs, axis=2), S, heads


@pytest.mark.parametrize("masked", [True, False])
@pytest.mark.parametrize("normalize", [False, True])
def test_mq_decode_equals_heads_with_broadcast_keys(masked, normalize):
    """A group sharing one key moment gives exactly the outputs of independent heads that
    all see the group's key and value: against the pair sum on the broadcast inputs."""
    group, Hk = 3, 2
    r = np.random.default_rng(70)
    q = r.standard_normal((2, Hk * group, 7, 4)) / 2
    k = r.standard_normal((2, Hk, 7, 4)) / 2
    v = r.standard_normal((2, Hk, 7, 3))
    if normalize:
        q, k = np.abs(q) + 0.1, np.abs(k) + 0.1
    gam = [0.9, 0.97]
    o, S, heads = _mq_run(q, k, v, gam, group, normalize, masked)
    kb, vb = np.repeat(k, group, axis=1), np.repeat(v, group, axis=1)
    gb = np.repeat(gam, group)
    ref = O.brute_force_forward(q, kb, vb, gb, normalize=normalize, masked=masked)
    assert rel(o, ref) < 1e-12
    _, st = O.serial_forward(q, kb, vb, gb, return_state=True)
    for j in range(Hk):
        for i in range(group):
            assert rel(S[:, j], st["S"][:, j * group + i]) < 1e-13
    for key in ("C", "G", "m", "h"):
        assert rel(heads[key], st[key]) < 1e-12


def test_mq_planted_mistake_is_caught():
    """Advancing the shared S once per head instead of once per group is caught."""
    group, Hk = 2, 1
    r = np.random.default_rng(71)
    q = r.standard_normal((1, group, 6, 3))
    k = r.standard_normal((1, Hk, 6, 3))
    v = r.standard_normal((1, Hk, 6, 2))
    ref = O.brute_force_forward(q, np.repeat(k, group, axis=1), np.repeat(v, group, axis=1), [0.9, 0.9])

    def per_head_update(S, heads, q_t, k_t, v_t, gamma, group_, normalize, eps, masked):
        S2 = S
        for _ in range(group_ - 1):  # the mistake: one extra update per additional head
            S2 = 0.9 * S2 + np.einsum("nja,njb->njab", k_t, k_t)
        return O.mq_decode_step(S2, heads, q_t, k_t, v_t, gamma, group_, normalize, eps, masked)

    bad, _, _ = _mq_run(q, k, v, [0.9], group, S_step=per_head_update)
    assert rel(bad, ref) > 1e-3
