"""Pins of the AHLA oracle (``oracle/ahla_oracle.py``) to what the pages and the mathematics
fix: closed forms, the masked matrix form of the operator, brute force, the chunked scan,
the combine's algebra, causality, and planted mistakes that each of these catches."""
import numpy as np
import pytest

from oracle import ahla_oracle as A


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


@pytest.mark.parametrize("g", [1.0, 0.8])
def test_closed_forms_n1_n2(g):
    q, k, v = rnd(1, 1, 2, 3, 2, seed=1)
    o = A.serial_forward(q, k, v, [g])[0, 0]
    Q, K, V = q[0, 0], k[0, 0], v[0, 0]
    assert np.allclose(o[0], (Q[0] @ K[0]) ** 2 * V[0], rtol=1e-13, atol=0)
    o2 = (g * (Q[1] @ K[0]) * (Q[0] @ K[0]) * V[0]      # j = 1, i = 1
          + g * (Q[1] @ K[1]) * (Q[1] @ K[0]) * V[0]    # j = 2, i = 1
          + (Q[1] @ K[1]) * (Q[1] @ K[1]) * V[1])       # j = 2, i = 2
    assert np.allclose(o[1], o2, rtol=1e-13, atol=0)


@pytest.mark.parametrize("g", [1.0, 0.9])
def test_masked_matrix_form(g):
    """O = L(A) (L(A) V), A = Q K^T, L keeping j <= t with weight g^(t-j): the left-cascaded
    product Q (K^T Q)(K^T V) of the technical summary with both causal masks (A1, A2)."""
    q, k, v = rnd(2, 1, 11, 4, 3, seed=2)
    for b in range(2):
        Q, K, V = q[b, 0], k[b, 0], v[b, 0]
        n = Q.shape[0]
        t, j = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
        L = np.where(j <= t, g ** (t - j).astype(float), 0.0) * (Q @ K.T)
        assert rel(A.serial_forward(q[b:b + 1], k[b:b + 1], v[b:b + 1], [g])[0, 0], L @ (L @ V)) < 1e-12


@pytest.mark.parametrize("normalize", [False, True])
def test_brute_force_equals_serial(normalize):
    q, k, v = rnd(1, 2, 9, 3, 2, seed=3, positive=normalize)
    g = [1.0, 0.85]
    assert rel(A.serial_forward(q, k, v, g, normalize), A.brute_force_forward(q, k, v, g, normalize)) < 1e-12


@pytest.mark.parametrize("chunk", [1, 2, 3, 5, 13])
def test_chunked_scan_equals_serial(chunk):
    q, k, v = rnd(1, 2, 13, 3, 2, seed=4)
    g = [0.9, 1.0]
    assert rel(A.chunked_scan_forward(q, k, v, g, chunk), A.serial_forward(q, k, v, g)) < 1e-12
    qp, kp, vp = rnd(1, 1, 10, 3, 2, seed=5, positive=True)
    assert rel(A.chunked_scan_forward(qp, kp, vp, [0.95], chunk, normalize=True),
               A.serial_forward(qp, kp, vp, [0.95], normalize=True)) < 1e-12


def _random_summary(r, d, dv):
    return {"P": r.standard_normal((d, dv)), "m": r.standard_normal(d), "E": r.standard_normal((d, dv)),
            "n": r.standard_normal(d), "R": r.standard_normal((d, d)), "rho": float(r.uniform(0.5, 1.0))}


def test_combine_is_associative_with_identity():
    r = np.random.default_rng(6)
    X, Y, Z = (_random_summary(r, 3, 2) for _ in range(3))
    left = A.combine(A.combine(X, Y), Z)
    right = A.combine(X, A.combine(Y, Z))
    for key in ("P", "m", "E", "n", "R"):
        assert rel(left[key], right[key]) < 1e-13
    e = A.identity_element(3, 2)
    for key in ("P", "m", "E", "n", "R"):
        assert np.array_equal(A.combine(e, X)[key], X[key]) and np.array_equal(A.combine(X, e)[key], X[key])


def test_causality_and_no_decay_reduction():
    q, k, v = rnd(1, 1, 12, 4, 3, seed=7)
    base = A.serial_forward(q, k, v, [0.9])
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[..., 7:, :] += 1.0
    k2[..., 7:, :] -= 0.5
    v2[..., 7:, :] *= 3.0
    assert np.array_equal(A.serial_forward(q2, k2, v2, [0.9])[..., :7, :], base[..., :7, :])
    assert np.array_equal(A.serial_forward(q, k, v, [1.0]), A.serial_forward(q, k, v, None))


def test_planted_mistakes_are_caught(monkeypatch):
    """Reading the inner product before P's update (dropping i == j), or decaying E twice
    (g^2 as for the symmetric variant's cross summaries), breaks brute-force agreement."""
    q, k, v = rnd(1, 1, 6, 3, 2, seed=8)
    ref = A.brute_force_forward(q, k, v, [0.9])

    def pre_update_inner(q_, k_, v_, gamma=None, normalize=False, eps=1e-6, return_state=False):
        qq, kk, vv = (np.asarray(x, dtype=np.float64) for x in (q_, k_, v_))
        g = 0.9
        P = np.zeros((3, 2))
        E = np.zeros((3, 2))
        out = np.zeros_like(vv)
        for t in range(qq.shape[2]):
            inner = qq[0, 0, t] @ P          # mistake: P before the token's own update
            P = g * P + np.outer(kk[0, 0, t], vv[0, 0, t])
            E = g * E + np.outer(kk[0, 0, t], inner)
            out[0, 0, t] = qq[0, 0, t] @ E
        return out

    assert rel(pre_update_inner(q, k, v), ref) > 1e-3
    brute_sq = A.brute_force_forward(q, k, v, [0.9 ** 2])  # g^2 per hop instead of g
    assert rel(brute_sq, ref) > 1e-3


def test_adjoint_matches_the_pair_sum_gradients():
    q, k, v = rnd(1, 2, 7, 3, 2, seed=20)
    dO = np.random.default_rng(21).standard_normal(v.shape)
    g = [0.9, 1.0]
    got = A.serial_backward(q, k, v, dO, g)
    ref = A.pairsum_grads(q, k, v, dO, g)
    for a, b in zip(got, ref):
        assert rel(a, b) < 1e-12


def test_adjoint_matches_central_differences():
    q, k, v = rnd(1, 1, 6, 3, 2, seed=22)
    dO = np.random.default_rng(23).standard_normal(v.shape)
    g = [0.85]
    dq, dk, dv = A.serial_backward(q, k, v, dO, g)
    loss = lambda q_, k_, v_: np.sum(A.serial_forward(q_, k_, v_, g) * dO)  # noqa: E731
    h = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = {"q": q, "k": k, "v": v}
            args_p[name], args_m[name] = xp, xm
            num[idx] = (loss(**{"q_": args_p["q"], "k_": args_p["k"], "v_": args_p["v"]})
                        - loss(**{"q_": args_m["q"], "k_": args_m["k"], "v_": args_m["v"]})) / (2 * h)
        assert rel(grad, num) < 1e-7, name


def test_adjoint_planted_mistake_is_caught():
    """Reading the inner adjoint from the pre-update E adjoint (dropping the token's own
    output term) breaks agreement with the pair-sum gradients."""
    q, k, v = rnd(1, 1, 5, 3, 2, seed=24)
    dO = np.random.default_rng(25).standard_normal(v.shape)
    ref = A.pairsum_grads(q, k, v, dO, [0.9])
    Q, K, V, O = q[0, 0], k[0, 0], v[0, 0], dO[0, 0]
    g = 0.9
    Ps, Es, Is = [], [], []
    P = np.zeros((3, 2))
    E = np.zeros((3, 2))
    for t in range(5):
        P = g * P + np.outer(K[t], V[t])
        i_t = Q[t] @ P
        E = g * E + np.outer(K[t], i_t)
        Ps.append(P); Es.append(E); Is.append(i_t)
    dk = np.zeros_like(K)
    Eb = np.zeros((3, 2))
    Pb = np.zeros((3, 2))
    for t in range(4, -1, -1):
        ib = Eb.T @ K[t]                           # mistake: before adding q_t dO_t^T
        Eb = g * Eb + np.outer(Q[t], O[t])
        dk[t] += Eb @ Is[t]
        Pb = g * Pb + np.outer(Q[t], ib)
        dk[t] += Pb @ V[t]
    assert rel(dk, ref[1][0, 0]) > 1e-3
