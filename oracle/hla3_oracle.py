"""Float64 CPU oracle for masked third-order Higher-order Linear Attention (HLA-3).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of
``bench.py`` may import it.  It shares no code with the CUDA library and never imports it.

Sources (page title, then the section on that page):
  [TS3] "Higher-order Linear Attention" -- technical summary, item "3. Dritte Ordnung HLA":
        third-order interactions defined by the matrix product A A^T A with A = Q K^T; the
        masked output keeps three primary prefix moments S^K, S^Q, P^KV and six cross
        summaries G^(1..3), h^(1..3) to enforce strict causality; the per-token update cost
        stays linear in the feature dimensions.
  [PS]  "Higher-order Linear Attention" -- section summary: the chunk scan of the
        third-order case is exact for gamma = 1; its segment maps are not printed.

Readings where the pages leave a step open (each is pinned by ``tests/test_hla3_oracle.py``):
  T1  The masked operator applies the causal mask to every factor and to the partial product
      of the first two, as the masked second-order output does for A A^T:
          O = ((A o M)(A o M)^T o M)(A o M) V,   M[t, s] = [s <= t],
      i.e.  o_t = sum_{j <= t} sum_{i <= j} sum_{l <= j} (q_t.k_i)(k_i.q_j)(q_j.k_l) v_l.
      Removing the terms with i > j or l > j from the full product q_t^T S^K S^Q P^KV takes
      three corrections by inclusion-exclusion ([i > j], [l > j], both), which is the count
      of cross summaries G^(1..3) the pages give, and three more, h^(1..3), for the
      denominator (v -> 1).
  T2  gamma = 1 only: the pages state the scan for that case.
  T3  Denominator den_t = the same triple sum with v_l replaced by 1; the normalised output is
      o_t / (den_t + eps).
  T4  Streaming form: with p_t = S^K_t q_t and u_t = P_t^T q_t (the first-order linear
      attention output at t),  Y_t = Y_{t-1} + p_t u_t^T  and  o_t = q_t^T Y_t.  This is the
      masked second-order output with the values v replaced by u (the "values" of the outer
      pair are the first-order outputs), which the GPU path evaluates as two passes.

Array conventions: q, k [B, H, n, d]; v [B, H, n, dv].
"""
from __future__ import annotations

import numpy as np

__all__ = ["brute_force_forward", "serial_forward", "matrix_form_forward", "first_order_forward", "state_floats",
           "decode_step"]


def _f64(*xs):
    return tuple(np.asarray(x, dtype=np.float64) for x in xs)


def brute_force_forward(q, k, v, normalize=False, eps=1e-6):
    """The triple sum of reading T1 (and T3), term by term.  O(n^4 d) per head: tiny n only."""
    q, k, v = _f64(q, k, v)
    B, H, n, d = q.shape
    dv = v.shape[-1]
    out = np.zeros((B, H, n, dv))
    for b in range(B):
        for h in range(H):
            A = q[b, h] @ k[b, h].T  # A[t, s] = q_t . k_s
            for t in range(n):
                num = np.zeros(dv)
                den = 0.0
                for j in range(t + 1):
                    for i in range(j + 1):
                        for l in range(j + 1):
                            w = A[t, i] * A[j, i] * A[j, l]
                            num += w * v[b, h, l]
                            den += w
                out[b, h, t] = num / (den + eps) if normalize else num
    return out


def matrix_form_forward(q, k, v, normalize=False, eps=1e-6):
    """Reading T1 as masked matrix products: ((A o M)(A o M)^T o M)(A o M) V."""
    q, k, v = _f64(q, k, v)
    B, H, n, d = q.shape
    M = np.tril(np.ones((n, n)))
    out = np.zeros(v.shape)
    for b in range(B):
        for h in range(H):
            Am = (q[b, h] @ k[b, h].T) * M
            W = ((Am @ Am.T) * M) @ Am
            o = W @ v[b, h]
            if normalize:
                o = o / (W.sum(axis=1) + eps)[:, None]
            out[b, h] = o
    return out


def first_order_forward(q, k, v):
    """Masked first-order linear attention, u_t = sum_{l <= t} (q_t . k_l) v_l, serially."""
    q, k, v = _f64(q, k, v)
    B, H, n, d = q.shape
    P = np.zeros((B, H, d, v.shape[-1]))
    out = np.zeros(v.shape)
    for t in range(n):
        P = P + np.einsum("bha,bhe->bhae", k[:, :, t], v[:, :, t])
        out[:, :, t] = np.einsum("bha,bhae->bhe", q[:, :, t], P)
    return out


def serial_forward(q, k, v, normalize=False, eps=1e-6):
    """Streaming form of reading T4: per token, S^K += k k^T and P^KV += k v^T (and the key
    mass m^K += k for the denominator), then Y += (S^K q)(P^T q)^T and o = q^T Y."""
    q, k, v = _f64(q, k, v)
    B, H, n, d = q.shape
    dv = v.shape[-1]
    S = np.zeros((B, H, d, d))
    P = np.zeros((B, H, d, dv))
    m = np.zeros((B, H, d))
    Y = np.zeros((B, H, d, dv))
    y = np.zeros((B, H, d))
    out = np.zeros((B, H, n, dv))
    for t in range(n):
        qt, kt, vt = q[:, :, t], k[:, :, t], v[:, :, t]
        S = S + np.einsum("bha,bhc->bhac", kt, kt)
        P = P + np.einsum("bha,bhe->bhae", kt, vt)
        m = m + kt
        p = np.einsum("bhac,bhc->bha", S, qt)           # S^K_t q_t
        u = np.einsum("bha,bhae->bhe", qt, P)           # P_t^T q_t
        Y = Y + np.einsum("bha,bhe->bhae", p, u)
        y = y + p * np.einsum("bha,bha->bh", qt, m)[..., None]
        o = np.einsum("bha,bhae->bhe", qt, Y)
        if normalize:
            o = o / (np.einsum("bha,bha->bh", qt, y) + eps)[..., None]
        out[:, :, t] = o
    return out


def state_floats(d, dv):
    """Floats of one head's streaming state [S^K d*d | P^KV d*dv | Y d*dv | m^K d | y d]."""
    return d * d + 2 * d * dv + 2 * d


def decode_step(state, q_t, k_t, v_t, normalize=False, eps=1e-6):
    """One streaming step of reading T4 on packed states [N, H, state_floats] (float64,
    updated in place): S^K += k k^T, P^KV += k v^T, m^K += k, then with p = S^K q and
    u = P^T q: Y += p u^T, y += p (q . m^K), o = q^T Y (/ (q^T y + eps)).  Returns o [N,H,dv]."""
    q_t, k_t, v_t = _f64(q_t, k_t, v_t)
    N, H, d = q_t.shape
    dv = v_t.shape[-1]
    o = 0
    S = state[..., o:o + d * d].reshape(N, H, d, d); o += d * d
    P = state[..., o:o + d * dv].reshape(N, H, d, dv); o += d * dv
    Y = state[..., o:o + d * dv].reshape(N, H, d, dv); o += d * dv
    m = state[..., o:o + d]; o += d
    y = state[..., o:o + d]
    S += np.einsum("nha,nhc->nhac", k_t, k_t)
    P += np.einsum("nha,nhe->nhae", k_t, v_t)
    m += k_t
    p = np.einsum("nhac,nhc->nha", S, q_t)
    u = np.einsum("nha,nhae->nhe", q_t, P)
    Y += np.einsum("nha,nhe->nhae", p, u)
    y += p * np.einsum("nha,nha->nh", q_t, m)[..., None]
    out = np.einsum("nha,nhae->nhe", q_t, Y)
    if normalize:
        out = out / (np.einsum("nha,nha->nh", q_t, y) + eps)[..., None]
    return out
