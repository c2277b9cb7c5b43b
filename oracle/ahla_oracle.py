"""Float64 CPU oracle for Asymmetric Higher-order Linear Attention (AHLA).

TEST INFRASTRUCTURE ONLY.  Like ``hla2_oracle``, this is the independent reference the
CUDA path is checked against: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
legs of ``bench.py`` may import it, and it shares no code with the CUDA library.

Sources (page title, then the section on that page):
  [TS2] "Higher-order Linear Attention" -- technical summary, item "2. Asymmetrische
        Lineare Aufmerksamkeit hoeherer Ordnung (AHLA)": the operator Q (K^T Q) (K^T V),
        values weighted in a single pass routed through an intermediate key index, with
        the streaming summaries P^KV_t, m^K_t, E_t, n_t and linear cost per token.
  [PS6] same title -- section summary §6 (left-cascaded product, strictly causal
        streaming), §6.1 (masked streaming identity with O(d dv) time and O(d dv + d) state
        per head; chunk summaries additionally use O(d^2) memory), §6.2 (exclusive
        associative scan plus local inclusion reproduces the serial recurrence), §6.3
        (optional decay and denominator normalisation).

Readings where the pages leave a step open (each pinned by ``tests/test_ahla_oracle.py``):
  A1  Masked operator: o_t = sum_{j <= t} sum_{i <= j} (q_t . k_j)(q_j . k_i) v_i, the
      product Q (K^T Q)(K^T V) with both causal masks keeping "on and before" (as for the
      symmetric HLA).  Unmasked, it is exactly [TS2]'s operator.
  A2  Decay: each hop attenuates by its distance, so pair (j, i) of output t carries
      g^((t-j) + (j-i)) = g^(t-i); every summary decays by g per token.
  A3  Summaries ([TS2] names): P^KV_t = g P^KV_{t-1} + k_t v_t^T,
      m^K_t = g m^K_{t-1} + k_t, E_t = g E_{t-1} + k_t (q_t^T P^KV_t),
      n_t = g n_{t-1} + k_t (q_t . m^K_t); o_t = q_t^T E_t, den_t = q_t^T n_t,
      normalised output o_t / (den_t + eps).  The inner read q_t^T P^KV_t uses the
      updated P (i == j kept), and E is read after its update (j == t kept).
  A4  Segment summary for the scan ([PS6] §6.1, the extra O(d^2) memory):
      R = sum_j k_j q_j^T over the segment, undecayed (the decays of a cross pair
      telescope to the later segment's attenuation rho = g^len, see A5).
  A5  Combine, A earlier, rho = g^len(B):
        P = rho P_A + P_B,  m = rho m_A + m_B,  R = R_A + R_B,
        E = rho E_A + E_B + rho R_B P_A,  n = rho n_A + n_B + rho R_B m_A.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "serial_forward",
    "brute_force_forward",
    "token_delta",
    "identity_element",
    "combine",
    "chunked_scan_forward",
    "serial_backward",
    "pairsum_grads",
]


def _gamma(gamma, H):
    if gamma is None:
        return np.ones(H)
    g = np.asarray(gamma, dtype=np.float64).reshape(-1)
    return np.full(H, g[0]) if g.size == 1 and H != 1 else g.reshape(H)


def serial_forward(q, k, v, gamma=None, normalize=False, eps=1e-6, return_state=False):
    """Streaming recurrence A3 over all tokens ([PS6] §6.1, §6.3)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, n, d = q.shape
    dv = v.shape[-1]
    g = _gamma(gamma, H)[None, :]
    P = np.zeros((B, H, d, dv))
    E = np.zeros((B, H, d, dv))
    m = np.zeros((B, H, d))
    nn = np.zeros((B, H, d))
    out = np.zeros((B, H, n, dv))
    for t in range(n):
        qt, kt, vt = q[:, :, t], k[:, :, t], v[:, :, t]
        P = g[..., None, None] * P + kt[..., :, None] * vt[..., None, :]
        m = g[..., None] * m + kt
        inner = np.einsum("bhd,bhde->bhe", qt, P)
        E = g[..., None, None] * E + kt[..., :, None] * inner[..., None, :]
        nn = g[..., None] * nn + kt * np.einsum("bhd,bhd->bh", qt, m)[..., None]
        o = np.einsum("bhd,bhde->bhe", qt, E)
        if normalize:
            o = o / (np.einsum("bhd,bhd->bh", qt, nn)[..., None] + eps)
        out[:, :, t] = o
    if return_state:
        return out, {"P": P, "E": E, "m": m, "n": nn}
    return out


def brute_force_forward(q, k, v, gamma=None, normalize=False, eps=1e-6):
    """The masked pair sum A1 with decay A2, term by term.  O(n^3) per head: tiny n only."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, n, d = q.shape
    dv = v.shape[-1]
    g = _gamma(gamma, H)
    out = np.zeros((B, H, n, dv))
    for b in range(B):
        for h in range(H):
            Q, K, V = q[b, h], k[b, h], v[b, h]
            for t in range(n):
                acc = np.zeros(dv)
                den = 0.0
                for j in range(t + 1):
                    a_tj = Q[t] @ K[j]
                    for i in range(j + 1):
                        w = g[h] ** (t - i) * a_tj * (Q[j] @ K[i])
                        acc += w * V[i]
                        den += w
                out[b, h, t] = acc / (den + eps) if normalize else acc
    return out


def token_delta(q_t, k_t, v_t, g):
    """Summary of a one-token segment (A3 from the empty prefix, A4): P = k v^T, m = k,
    E = k (q^T P) = (q . k) k v^T, n = (q . k) k, R = k q^T, attenuation g."""
    qk = float(q_t @ k_t)
    return {"P": np.outer(k_t, v_t), "m": k_t.copy(), "E": qk * np.outer(k_t, v_t), "n": qk * k_t,
            "R": np.outer(k_t, q_t), "rho": float(g)}


def identity_element(d, dv):
    """The empty segment: every summary zero, attenuation 1."""
    return {"P": np.zeros((d, dv)), "m": np.zeros(d), "E": np.zeros((d, dv)), "n": np.zeros(d),
            "R": np.zeros((d, d)), "rho": 1.0}


def combine(A, B):
    """Combine A5 of segment summaries, A earlier ([PS6] §6.2)."""
    r = B["rho"]
    return {"P": r * A["P"] + B["P"], "m": r * A["m"] + B["m"], "R": A["R"] + B["R"],
            "E": r * A["E"] + B["E"] + r * (B["R"] @ A["P"]),
            "n": r * A["n"] + B["n"] + r * (B["R"] @ A["m"]),
            "rho": A["rho"] * r}


def chunked_scan_forward(q, k, v, gamma=None, chunk=16, normalize=False, eps=1e-6):
    """Chunk-parallel form ([PS6] §6.2): token deltas combined inside each chunk by an
    exclusive scan, an exclusive scan of the chunk totals gives each chunk's carry-in,
    and each token's inclusive state is carry (+) exclusive prefix (+) its delta; the
    output is read from that state as in A3."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, n, d = q.shape
    dv = v.shape[-1]
    g = _gamma(gamma, H)
    out = np.zeros((B, H, n, dv))
    for b in range(B):
        for h in range(H):
            deltas = [token_delta(q[b, h, t], k[b, h, t], v[b, h, t], g[h]) for t in range(n)]
            chunks = [deltas[s:s + chunk] for s in range(0, n, chunk)]
            totals = []
            for c in chunks:
                tot = identity_element(d, dv)
                for dl in c:
                    tot = combine(tot, dl)
                totals.append(tot)
            carry = identity_element(d, dv)
            t = 0
            for ci, c in enumerate(chunks):
                prefix = identity_element(d, dv)
                for dl in c:
                    st = combine(combine(carry, prefix), dl)
                    o = q[b, h, t] @ st["E"]
                    if normalize:
                        o = o / (q[b, h, t] @ st["n"] + eps)
                    out[b, h, t] = o
                    prefix = combine(prefix, dl)
                    t += 1
                carry = combine(carry, totals[ci])
    return out


def serial_backward(q, k, v, dout, gamma=None):
    """Hand adjoint of the unnormalised recurrence A3 ([PS] §4.2 states the reverse-mode scan
    for the second-order case; the same reverse sweep applies here).

    Forward at token t:  P_t = g P + k v^T;  i_t = P_t^T q;  E_t = g E + k i_t^T;  o_t = E_t^T q.
    Reverse sweep with state adjoints (Eb, Pb) flowing from t+1 to t:
        Eb = g Eb + q dO^T;        dq += E_t dO;
        ib = Eb^T k;               dk += Eb i_t;
        Pb = g Pb + q ib^T;        dq += P_t ib;
        dk += Pb v;                dv += Pb^T k.
    Returns (dq, dk, dv) in float64."""
    q, k, v, dout = (np.asarray(x, dtype=np.float64) for x in (q, k, v, dout))
    B, H, n, d = q.shape
    dv_ = v.shape[-1]
    g = _gamma(gamma, H)[None, :]
    Ps, Es, Is = [], [], []
    P = np.zeros((B, H, d, dv_))
    E = np.zeros((B, H, d, dv_))
    for t in range(n):  # forward, keeping the states
        P = g[..., None, None] * P + np.einsum("bha,bhe->bhae", k[:, :, t], v[:, :, t])
        inner = np.einsum("bha,bhae->bhe", q[:, :, t], P)
        E = g[..., None, None] * E + np.einsum("bha,bhe->bhae", k[:, :, t], inner)
        Ps.append(P)
        Es.append(E)
        Is.append(inner)
    dq, dk, dvv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    Eb = np.zeros((B, H, d, dv_))
    Pb = np.zeros((B, H, d, dv_))
    for t in range(n - 1, -1, -1):
        qt, kt, vt, ot = q[:, :, t], k[:, :, t], v[:, :, t], dout[:, :, t]
        Eb = g[..., None, None] * Eb + np.einsum("bha,bhe->bhae", qt, ot)
        dq[:, :, t] += np.einsum("bhae,bhe->bha", Es[t], ot)
        ib = np.einsum("bhae,bha->bhe", Eb, kt)
        dk[:, :, t] += np.einsum("bhae,bhe->bha", Eb, Is[t])
        Pb = g[..., None, None] * Pb + np.einsum("bha,bhe->bhae", qt, ib)
        dq[:, :, t] += np.einsum("bhae,bhe->bha", Ps[t], ib)
        dk[:, :, t] += np.einsum("bhae,bhe->bha", Pb, vt)
        dvv[:, :, t] += np.einsum("bhae,bha->bhe", Pb, kt)
    return dq, dk, dvv


def pairsum_grads(q, k, v, dout, gamma=None):
    """Gradients of L = sum_t dO_t . o_t with o_t the pair sum A1 (decay A2), differentiated
    term by term: each term g^(t-i) (q_t.k_j)(q_j.k_i) v_i contributes to q_t, k_j, q_j, k_i
    and v_i.  O(n^3) per head: tiny n only."""
    q, k, v, dout = (np.asarray(x, dtype=np.float64) for x in (q, k, v, dout))
    B, H, n, d = q.shape
    g = _gamma(gamma, H)
    dq, dk, dvv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            Q, K, V, O = q[b, h], k[b, h], v[b, h], dout[b, h]
            for t in range(n):
                for j in range(t + 1):
                    for i in range(j + 1):
                        w = g[h] ** (t - i)
                        a, c = Q[t] @ K[j], Q[j] @ K[i]
                        s = O[t] @ V[i]  # dL/d(weight of the term)
                        dq[b, h, t] += w * s * c * K[j]
                        dk[b, h, j] += w * s * c * Q[t]
                        dq[b, h, j] += w * s * a * K[i]
                        dk[b, h, i] += w * s * a * Q[j]
                        dvv[b, h, i] += w * a * c * O[t]
    return dq, dk, dvv
