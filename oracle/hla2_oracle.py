"""Float64 CPU oracle for masked second-order Higher-order Linear Attention (HLA-2).

TEST INFRASTRUCTURE ONLY.  This module is the independent reference that the CUDA
path is checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.  It shares
no code, table or helper with the CUDA library and never imports it.

Sources (page title, then the section or formula on that page):
  [TS]  "Higher-order Linear Attention" -- technical summary ("Technische Zusammenfassung"),
        item "1. Zweite Ordnung HLA": prefix moments S^K_t = sum_{i<=t} k_i k_i^T,
        C^QV_t = sum_{i<=t} q_i v_i^T, m^Q_t = sum_{i<=t} q_i; the extended summaries
        G_t, h_t that remove the future terms of the naive product S^K_t C^QV_t; the
        output o_t = q_t^T (S^K_t C^QV_t - G_t); a ratio-normalised variant that divides
        by a masked denominator built the same way.
  [TS4] same page, item "4. Paralleles Training durch assoziative Scans": semidirect
        product that carries the cross term S^K_B C^QV_A; exclusive Blelloch scan over
        segment summaries reproduces the serial recurrence exactly.
  [PS]  "Higher-order Linear Attention" -- section summary: §2 (row-vector outputs,
        unnormalised vs ratio-normalised), §2.1 (causal mask keeps j <= t), §3.1 (two
        extra summaries, O(d^2 + d dv) per token), §4.1 (token deltas, inclusive state =
        exclusive prefix combined with the token delta, segments composed in time
        order), §4.2 (masked semidirect product, tuple (S, C, m, G, h); reverse-mode scan
        gives the serial recurrence's gradients), §4 (exclusive Blelloch scan inside a
        chunk, then a scan of chunk summaries for the carry-in), §4.3 (fixed
        exponential decay: segment summaries carry one attenuation factor and the
        updates are the decayed analogues of the online ones), §5.1 (default output is
        unnormalised; optional normalisation divides by the masked denominator).

Readings where the pages leave a step open (each is pinned by a test in
``tests/test_oracle.py``):
  R1  G and h are updated from the PRE-update C and m:
        G_t = g^2 G_{t-1} + g k_t (k_t^T C_{t-1}),  h_t = g^2 h_{t-1} + g k_t (k_t^T m_{t-1}).
      This removes exactly the pairs (key index i) > (value index j) from S_t C_t, so the
      diagonal pair i == j is kept ([PS] §2.1, "on and before").
  R2  Decay g in (0, 1]: S, C, m decay by g per token; G and h by g^2.  Equivalently
      every pair (i <= j <= t) carries weight g^((t-i) + (t-j)), and the combine uses
      one attenuation factor rho = g^len per segment ([PS] §4.3).
  R3  No feature map: C = sum q v^T with the raw query ([TS]).
  R4  Denominator den_t = q_t^T (S_t m_t - h_t); normalised output o_t / (den_t + eps).
  R5  Row-vector convention: o_t has dv entries ([PS] §2).
  R6  Unmasked variant ([PS] §3, the "numerator-style bilinear form"; [PS] §4.1): the
      output is the naive product o_t = q_t^T S_t C_t (every pair i, j <= t, weight
      g^((t-i) + (t-j))), normalised by q_t^T S_t m_t.  Its scan carries only (S, C, m)
      and combines them by decayed addition, with no cross term (the unmasked monoid).
      The state's G and h play no part in it; the unmasked chunked scan reports them as 0.
  R7  Multi-query sharing ([PS] §5.2: it cuts the state from O(h d^2) to O(d^2 + h d dv)):
      the heads of a group share the key and the value of each token, so they share S^K (one
      per group, with one decay per group); C, G, m, h stay per head because they carry each
      head's own query.

Array conventions: q, k [B, H, n, d]; v, dout [B, H, n, dv]; gamma [H] (None means 1).
State dict per head: S [B,H,d,d], C [B,H,d,dv], m [B,H,d], G [B,H,d,dv], h [B,H,d].
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "zero_state",
    "step",
    "serial_forward",
    "brute_force_forward",
    "token_delta",
    "identity_element",
    "combine",
    "blelloch_exclusive_scan",
    "chunked_scan_forward",
    "unmasked_delta",
    "unmasked_identity",
    "combine_unmasked",
    "mq_decode_step",
    "serial_backward",
    "serial_backward_normalized",
    "pairsum_grads",
    "pack_state",
    "unpack_state",
    "state_floats",
    "compact_state_floats",
    "compact_from_state",
    "state_from_compact",
]


def _gamma(gamma, H):
    if gamma is None:
        return np.ones(H, dtype=np.float64)
    g = np.asarray(gamma, dtype=np.float64).reshape(H)
    if np.any(g <= 0.0) or np.any(g > 1.0):
        raise ValueError("decay must lie in (0, 1]")
    return g


def zero_state(B, H, d, dv):
    """The empty prefix: every summary is zero ([PS] §4.1 identity of the monoid)."""
    z = np.zeros
    return {
        "S": z((B, H, d, d)),
        "C": z((B, H, d, dv)),
        "m": z((B, H, d)),
        "G": z((B, H, d, dv)),
        "h": z((B, H, d)),
    }


def step(state, q_t, k_t, v_t, g, normalize=False, eps=1e-6, masked=True):
    """One online update followed by the masked output ([TS], [PS] §3.1; readings R1-R4),
    or with ``masked=False`` the unmasked one, q^T S C (reading R6).

    q_t, k_t [B,H,d]; v_t [B,H,dv]; g [H].  Returns (new_state, o_t) with o_t [B,H,dv].
    The state is updated in the order the definitions require: G and h first (they
    read the old C and m), then S, C, m.  The output uses the updated state.
    """
    gg = g[None, :]
    S, C, m, G, h = state["S"], state["C"], state["m"], state["G"], state["h"]
    # k^T C_{t-1} and k^T m_{t-1}: the cross-summaries see only earlier values
    kC = np.einsum("bha,bhae->bhe", k_t, C)
    km = np.einsum("bha,bha->bh", k_t, m)
    G = (gg * gg)[..., None, None] * G + gg[..., None, None] * np.einsum("bha,bhe->bhae", k_t, kC)
    h = (gg * gg)[..., None] * h + gg[..., None] * k_t * km[..., None]
    S = gg[..., None, None] * S + np.einsum("bha,bhc->bhac", k_t, k_t)
    C = gg[..., None, None] * C + np.einsum("bha,bhe->bhae", q_t, v_t)
    m = gg[..., None] * m + q_t
    # o_t = q^T (S C - G), evaluated as (q^T S) C - q^T G so S C is never formed
    u = np.einsum("bha,bhac->bhc", q_t, S)
    o = np.einsum("bhc,bhce->bhe", u, C)
    if masked:
        o = o - np.einsum("bha,bhae->bhe", q_t, G)
    if normalize:
        den = np.einsum("bhc,bhc->bh", u, m)
        if masked:
            den = den - np.einsum("bha,bha->bh", q_t, h)
        o = o / (den + eps)[..., None]
    return {"S": S, "C": C, "m": m, "G": G, "h": h}, o


def serial_forward(q, k, v, gamma=None, normalize=False, eps=1e-6, init_state=None,
                   return_state=False, masked=True):
    """Serial recurrence over all tokens: the streaming form of [TS] / [PS] §3.1 (with
    ``masked=False`` the unmasked output of reading R6; the state evolves the same way)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, n, d = q.shape
    dv = v.shape[-1]
    g = _gamma(gamma, H)
    st = zero_state(B, H, d, dv) if init_state is None else {
        key: np.array(val, dtype=np.float64, copy=True) for key, val in init_state.items()}
    out = np.zeros((B, H, n, dv))
    for t in range(n):
        st, out[:, :, t] = step(st, q[:, :, t], k[:, :, t], v[:, :, t], g, normalize, eps, masked)
    return (out, st) if return_state else out


def brute_force_forward(q, k, v, gamma=None, normalize=False, eps=1e-6, masked=True):
    """The masked second-order output written as its pair sum (readings R1, R2):

        o_t = sum_{j <= t} sum_{i <= j} g^((t-i)+(t-j)) (q_t . k_i)(k_i . q_j) v_j

    i.e. the strictly causal mask of [PS] §2.1 applied to the bilinear form
    q_t^T S_t C_t of [TS], keeping key index i at or before value index j.  With
    ``masked=False`` i runs to t instead (reading R6: the whole product q_t^T S_t C_t).
    The denominator is the same sum with v_j replaced by 1.  O(n^3) per head: tiny n only.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, n, d = q.shape
    dv = v.shape[-1]
    g = _gamma(gamma, H)
    out = np.zeros((B, H, n, dv))
    for b in range(B):
        for hh in range(H):
            A = q[b, hh] @ k[b, hh].T          # A[t, i] = q_t . k_i
            for t in range(n):
                num = np.zeros(dv)
                den = 0.0
                for j in range(t + 1):
                    w = 0.0
                    for i in range(j + 1 if masked else t + 1):
                        w += g[hh] ** ((t - i) + (t - j)) * A[t, i] * A[j, i]
                    num += w * v[b, hh, j]
                    den += w
                out[b, hh, t] = num / (den + eps) if normalize else num
    return out


# ---------------------------------------------------------------------------
# Scan algebra ([PS] §4.1-§4.3, [TS4])
# ---------------------------------------------------------------------------

def token_delta(q_t, k_t, v_t, g):
    """Per-token delta ([PS] §4.1): (k k^T, q v^T, q, 0, 0) with attenuation rho = g.

    Arguments are single-head vectors; g is a scalar.  The cross summaries of one
    token are zero: a single token has no (later key, earlier value) pair.
    """
    d, dv = k_t.shape[0], v_t.shape[0]
    return {
        "S": np.outer(k_t, k_t),
        "C": np.outer(q_t, v_t),
        "m": np.array(q_t, dtype=np.float64),
        "G": np.zeros((d, dv)),
        "h": np.zeros(d),
        "rho": float(g),
    }


def identity_element(d, dv):
    """Neutral element of the combine: empty segment, attenuation 1."""
    return {"S": np.zeros((d, d)), "C": np.zeros((d, dv)), "m": np.zeros(d),
            "G": np.zeros((d, dv)), "h": np.zeros(d), "rho": 1.0}


def combine(A, B):
    """Masked semidirect product A (+) B, A the earlier segment ([PS] §4.2, §4.3; [TS4]).

    With rho = rho_B (B's attenuation, g^len(B)):
        S = rho S_A + S_B          C = rho C_A + C_B          m = rho m_A + m_B
        G = rho^2 G_A + G_B + rho S_B C_A      (cross term S^K_B C^QV_A of [TS4])
        h = rho^2 h_A + h_B + rho S_B m_A
        rho_AB = rho_A rho_B
    The cross term collects the pairs whose key lies in B and value in A (key after
    value), which the mask removes; rho^2 on G_A and the single rho on the cross term
    follow from the pair weight g^((t-i)+(t-j)) of reading R2.
    """
    r = B["rho"]
    return {
        "S": r * A["S"] + B["S"],
        "C": r * A["C"] + B["C"],
        "m": r * A["m"] + B["m"],
        "G": r * r * A["G"] + B["G"] + r * (B["S"] @ A["C"]),
        "h": r * r * A["h"] + B["h"] + r * (B["S"] @ A["m"]),
        "rho": A["rho"] * B["rho"],
    }


def unmasked_delta(q_t, k_t, v_t, g):
    """Token delta of the unmasked monoid ([PS] §4.1; reading R6): (k k^T, q v^T, q)
    with attenuation g."""
    return {"S": np.outer(k_t, k_t), "C": np.outer(q_t, v_t),
            "m": np.array(q_t, dtype=np.float64), "rho": float(g)}


def unmasked_identity(d, dv):
    """Neutral element of the unmasked monoid: empty segment, attenuation 1."""
    return {"S": np.zeros((d, d)), "C": np.zeros((d, dv)), "m": np.zeros(d), "rho": 1.0}


def combine_unmasked(A, B):
    """Unmasked monoid ([PS] §4.1, with the decay of §4.3), A the earlier segment: each
    moment is the later segment's plus the earlier one's attenuated by rho_B, with no
    cross term, because the unmasked output keeps every (key, value) pair."""
    r = B["rho"]
    return {"S": r * A["S"] + B["S"], "C": r * A["C"] + B["C"], "m": r * A["m"] + B["m"],
            "rho": A["rho"] * B["rho"]}


def blelloch_exclusive_scan(items, d, dv, op=None, unit=None):
    """Exclusive Blelloch scan (up-sweep, then down-sweep) under ``combine`` ([PS] §4).

    The list is padded with identity elements to a power of two.  The operator is not
    commutative, so the down-sweep forms the right child's prefix as
    (parent prefix) (+) (left subtree total), keeping time order.
    Returns prefixes[t] = items[0] (+) ... (+) items[t-1] (identity for t = 0).
    ``op`` and ``unit`` default to the masked ``combine`` and ``identity_element``.
    """
    op = combine if op is None else op
    unit = identity_element if unit is None else unit
    n = len(items)
    if n == 0:
        return []
    size = 1
    while size < n:
        size *= 2
    tree = list(items) + [unit(d, dv) for _ in range(size - n)]
    # up-sweep: tree[right] becomes the total of its subtree
    stride = 1
    while stride < size:
        for right in range(2 * stride - 1, size, 2 * stride):
            left = right - stride
            tree[right] = op(tree[left], tree[right])
        stride *= 2
    # down-sweep
    tree[size - 1] = unit(d, dv)
    stride = size // 2
    while stride >= 1:
        for right in range(2 * stride - 1, size, 2 * stride):
            left = right - stride
            left_total = tree[left]
            tree[left] = tree[right]
            tree[right] = op(tree[right], left_total)
        stride //= 2
    return tree[:n]


def _output_from_state(st, q_t, normalize, eps, masked=True):
    """o_t = q^T (S C - G) and den_t = q^T (S m - h) on an inclusive state ([TS], R4);
    unmasked, q^T S C and q^T S m (R6)."""
    u = q_t @ st["S"]
    o = u @ st["C"] - (q_t @ st["G"] if masked else 0.0)
    if normalize:
        den = u @ st["m"] - (q_t @ st["h"] if masked else 0.0)
        o = o / (den + eps)
    return o


def chunked_scan_forward(q, k, v, gamma=None, chunk=16, normalize=False, eps=1e-6,
                         init_state=None, return_state=False, masked=True):
    """Chunk-parallel forward in the order the pages give it ([PS] §4, §5; [TS4]):

      1. split [n] into chunks of width ``chunk`` (the last one may be shorter);
      2. token deltas (§4.1);
      3. exclusive Blelloch scan of the deltas inside each chunk;
      4. chunk summaries (the total of each chunk) and an exclusive scan of them,
         seeded with the initial state, giving each chunk's carry-in;
      5. inclusive state of token t = carry (+) local prefix (+) delta_t;
      6. output from the inclusive state.

    ``masked=False`` runs the same steps in the unmasked monoid on (S, C, m) and forms the
    unmasked output (reading R6); its final state reports G = h = 0.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, n, d = q.shape
    dv = v.shape[-1]
    g = _gamma(gamma, H)
    out = np.zeros((B, H, n, dv))
    finals = zero_state(B, H, d, dv)
    if masked:
        delta, op, unit, keys = token_delta, combine, identity_element, ("S", "C", "m", "G", "h")
    else:
        delta, op, unit, keys = unmasked_delta, combine_unmasked, unmasked_identity, ("S", "C", "m")
    for b in range(B):
        for hh in range(H):
            deltas = [delta(q[b, hh, t], k[b, hh, t], v[b, hh, t], g[hh]) for t in range(n)]
            chunks = [deltas[s:s + chunk] for s in range(0, n, chunk)]
            local_prefix = [blelloch_exclusive_scan(c, d, dv, op, unit) for c in chunks]
            totals = [op(pre[-1], c[-1]) for c, pre in zip(chunks, local_prefix)]
            start = unit(d, dv)
            if init_state is not None:
                for key in keys:
                    start[key] = np.array(init_state[key][b, hh], dtype=np.float64)
            # exclusive scan of the chunk summaries; carry-in of chunk c = start (+) excl[c]
            excl = blelloch_exclusive_scan(totals, d, dv, op, unit)
            t = 0
            for ci, (c, pre) in enumerate(zip(chunks, local_prefix)):
                carry = op(start, excl[ci])
                for li in range(len(c)):
                    incl = op(op(carry, pre[li]), c[li])
                    out[b, hh, t] = _output_from_state(incl, q[b, hh, t], normalize, eps, masked)
                    t += 1
            fin = op(start, op(excl[-1], totals[-1])) if totals else start
            for key in keys:
                finals[key][b, hh] = fin[key]
    return (out, finals) if return_state else out


# ---------------------------------------------------------------------------
# Reverse mode ([PS] §4.2: the reverse-mode scan reproduces the serial gradients)
# ---------------------------------------------------------------------------

def serial_backward(q, k, v, dout, gamma=None):
    """Hand-derived adjoint of the unnormalised serial recurrence of ``step``.

    Forward at token t (reading R1, R2):
        G_t = g^2 G_{t-1} + g k (k^T C_{t-1});  S_t = g S_{t-1} + k k^T;
        C_t = g C_{t-1} + q v^T;  u_t = S_t^T q;  o_t = C_t^T u_t - G_t^T q.
    Reverse sweep with state adjoints (Sb, Cb, Gb) flowing from t+1 to t:
        Cb += u dO^T;  ub = C_t dO;  Sb += q ub^T;  Gb -= q dO^T;
        dq += S_t ub - G_t dO;
        then through the updates:  r = C_{t-1}^T k,  rb = g Gb^T k,
        dk += g Gb r + C_{t-1} rb + (Sb + Sb^T) k;  dq += Cb v;  dv += Cb^T q;
        Cb_{t-1} = g Cb + k rb^T;  Sb_{t-1} = g Sb;  Gb_{t-1} = g^2 Gb.
    All per-token states are recomputed forward first and kept (tiny/medium n only).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    B, H, n, d = q.shape
    dv = v.shape[-1]
    g = _gamma(gamma, H)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dvv = np.zeros_like(v)
    for b in range(B):
        for hh in range(H):
            gh = g[hh]
            S = np.zeros((d, d))
            C = np.zeros((d, dv))
            G = np.zeros((d, dv))
            Ss, Cs, Gs, Cprev = [], [], [], []
            for t in range(n):
                qt, kt, vt = q[b, hh, t], k[b, hh, t], v[b, hh, t]
                Cprev.append(C.copy())
                G = gh * gh * G + gh * np.outer(kt, kt @ C)
                S = gh * S + np.outer(kt, kt)
                C = gh * C + np.outer(qt, vt)
                Ss.append(S.copy())
                Cs.append(C.copy())
                Gs.append(G.copy())
            Sb = np.zeros((d, d))
            Cb = np.zeros((d, dv))
            Gb = np.zeros((d, dv))
            for t in range(n - 1, -1, -1):
                qt, kt, vt, dOt = q[b, hh, t], k[b, hh, t], v[b, hh, t], dout[b, hh, t]
                S, C, G, Cp = Ss[t], Cs[t], Gs[t], Cprev[t]
                u = S.T @ qt
                # output o_t = C^T u - G^T q
                Cb = Cb + np.outer(u, dOt)
                ub = C @ dOt
                Sb = Sb + np.outer(qt, ub)
                Gb = Gb - np.outer(qt, dOt)
                dq[b, hh, t] += S @ ub - G @ dOt
                # G_t = g^2 G_{t-1} + g k r^T with r = C_{t-1}^T k
                r = Cp.T @ kt
                rb = gh * (Gb.T @ kt)
                dk[b, hh, t] += gh * (Gb @ r) + Cp @ rb
                # S_t = g S_{t-1} + k k^T
                dk[b, hh, t] += (Sb + Sb.T) @ kt
                # C_t = g C_{t-1} + q v^T
                dq[b, hh, t] += Cb @ vt
                dvv[b, hh, t] += Cb.T @ qt
                # adjoints of the previous state
                Cb = gh * Cb + np.outer(kt, rb)
                Sb = gh * Sb
                Gb = gh * gh * Gb
    return dq, dk, dvv


def serial_backward_normalized(q, k, v, dout, gamma=None, eps=1e-6):
    """Gradients of L = sum_t dO_t . o_t for the ratio-normalised output
    o_t = num_t / (den_t + eps) ([PS] §2, §5.1; reading R4), by the quotient rule:
        dnum_t = dO_t / (den_t + eps),   dden_t = -(dO_t . num_t) / (den_t + eps)^2.
    num is the unnormalised output and den the same pair sum with every v_j replaced by 1
    (R4).  Both are linear in v, so each path goes through the unnormalised adjoint
    ``serial_backward``: once with (v, dnum), once with (1, dden).  The second path
    contributes to dq and dk only.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    ones = np.ones(v.shape[:-1] + (1,))
    num = serial_forward(q, k, v, gamma)
    den = serial_forward(q, k, ones, gamma)[..., 0]
    inv = 1.0 / (den + eps)
    dnum = dout * inv[..., None]
    dden = -np.sum(dout * num, axis=-1) * inv * inv
    dq1, dk1, dv1 = serial_backward(q, k, v, dnum, gamma)
    dq2, dk2, _ = serial_backward(q, k, ones, dden[..., None], gamma)
    return dq1 + dq2, dk1 + dk2, dv1


def pairsum_grads(q, k, v, dout, gamma=None):
    """Gradients of L = sum_t dO_t . o_t taken term by term on the pair sum of
    ``brute_force_forward`` (unnormalised).  Each pair (i <= j <= t) with weight
    w = g^((t-i)+(t-j)) contributes w (q_t.k_i)(k_i.q_j)(v_j.dO_t), so
        dq_t += w (k_i.q_j)(v_j.dO_t) k_i,   dq_j += w (q_t.k_i)(v_j.dO_t) k_i,
        dk_i += w (v_j.dO_t) [ (k_i.q_j) q_t + (q_t.k_i) q_j ],
        dv_j += w (q_t.k_i)(k_i.q_j) dO_t.
    O(n^3) per head: tiny n only.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    B, H, n, d = q.shape
    g = _gamma(gamma, H)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dvv = np.zeros_like(v)
    for b in range(B):
        for hh in range(H):
            Q, K, V, dO = q[b, hh], k[b, hh], v[b, hh], dout[b, hh]
            for t in range(n):
                for j in range(t + 1):
                    vd = V[j] @ dO[t]
                    for i in range(j + 1):
                        w = g[hh] ** ((t - i) + (t - j))
                        a_ti = Q[t] @ K[i]
                        a_ji = Q[j] @ K[i]
                        dq[b, hh, t] += w * a_ji * vd * K[i]
                        dq[b, hh, j] += w * a_ti * vd * K[i]
                        dk[b, hh, i] += w * vd * (a_ji * Q[t] + a_ti * Q[j])
                        dvv[b, hh, j] += w * a_ti * a_ji * dO[t]
    return dq, dk, dvv


# ---------------------------------------------------------------------------
# Packed state layout of the decode step: per head [S d*d | C d*dv | G d*dv | m d | h d]
# ---------------------------------------------------------------------------

def state_floats(d, dv):
    return d * d + 2 * d * dv + 2 * d


def pack_state(st):
    """State dict -> [B, H, state_floats] float64 in the decode layout."""
    S, C, G, m, h = st["S"], st["C"], st["G"], st["m"], st["h"]
    B, H, d, _ = S.shape
    return np.concatenate([S.reshape(B, H, -1), C.reshape(B, H, -1), G.reshape(B, H, -1),
                           m.reshape(B, H, -1), h.reshape(B, H, -1)], axis=-1)


def unpack_state(flat, d, dv):
    flat = np.asarray(flat, dtype=np.float64)
    B, H, _ = flat.shape
    o = 0
    S = flat[..., o:o + d * d].reshape(B, H, d, d); o += d * d
    C = flat[..., o:o + d * dv].reshape(B, H, d, dv); o += d * dv
    G = flat[..., o:o + d * dv].reshape(B, H, d, dv); o += d * dv
    m = flat[..., o:o + d].reshape(B, H, d); o += d
    h = flat[..., o:o + d].reshape(B, H, d); o += d
    return {"S": S, "C": C, "m": m, "G": G, "h": h}


# ---------------------------------------------------------------------------
# Compact decode layout (a storage choice of the GPU library, not of the pages): S is a
# sum of decayed k k^T, hence symmetric, and only its upper block triangle is stored --
# row a keeps S[a, b] for b = 4 floor(a/4) .. d-1 -- followed by C, G, m, h.
# ---------------------------------------------------------------------------

def compact_state_floats(d, dv):
    return d * (d + 4) // 2 + 2 * d * dv + 2 * d


def compact_from_state(flat, d, dv):
    """[B, H, state_floats] packed states -> [B, H, compact_state_floats] (S's upper block
    triangle, row by row, then C, G, m, h)."""
    flat = np.asarray(flat, dtype=np.float64)
    S = flat[..., :d * d].reshape(flat.shape[:-1] + (d, d))
    rows = [S[..., a, 4 * (a // 4):] for a in range(d)]
    return np.concatenate(rows + [flat[..., d * d:]], axis=-1)


def state_from_compact(flat, d, dv):
    """Inverse of compact_from_state with S mirrored from the stored triangle."""
    flat = np.asarray(flat, dtype=np.float64)
    S = np.zeros(flat.shape[:-1] + (d, d))
    o = 0
    for a in range(d):
        b0 = 4 * (a // 4)
        S[..., a, b0:] = flat[..., o:o + d - b0]
        o += d - b0
    for a in range(d):
        for b in range(4 * (a // 4)):
            S[..., a, b] = S[..., b, a]
    return np.concatenate([S.reshape(flat.shape[:-1] + (d * d,)), flat[..., o:]], axis=-1)



# ---------------------------------------------------------------------------
# Multi-query sharing of the key moment ([PS] §5.2: with keys shared by a group of heads,
# S^K is shared and the state is O(d^2 + h d dv) per group; reading R7)
# ---------------------------------------------------------------------------

def mq_decode_step(S, heads, q_t, k_t, v_t, gamma, group, normalize=False, eps=1e-6, masked=True):
    """One decode step with one key moment per group of ``group`` query heads (reading R7).

    S [N, Hk, d, d] is shared by the heads g*group .. g*group+group-1 of key group g;
    heads = {"C": [N,H,d,dv], "G": [N,H,d,dv], "m": [N,H,d], "h": [N,H,d]} with
    H = Hk * group; q_t [N,H,d]; k_t [N,Hk,d] and v_t [N,Hk,dv] belong to the group;
    gamma None or [Hk] (one decay per group, since the shared S carries it).
    Returns (S, heads, o [N,H,dv]); the updates are those of ``step`` with the group's
    key and value, and S is advanced once per group.
    """
    S = np.array(S, dtype=np.float64, copy=True)
    hs = {key: np.array(val, dtype=np.float64, copy=True) for key, val in heads.items()}
    q_t = np.asarray(q_t, dtype=np.float64)
    k_t = np.asarray(k_t, dtype=np.float64)
    v_t = np.asarray(v_t, dtype=np.float64)
    N, Hk, d = k_t.shape
    dv = v_t.shape[-1]
    g = _gamma(gamma, Hk)
    out = np.zeros((N, Hk * group, dv))
    for b in range(N):
        for j in range(Hk):
            k, v, gj = k_t[b, j], v_t[b, j], g[j]
            S[b, j] = gj * S[b, j] + np.outer(k, k)
            for i in range(group):
                hh = j * group + i
                q = q_t[b, hh]
                C, G, m, h = hs["C"][b, hh], hs["G"][b, hh], hs["m"][b, hh], hs["h"][b, hh]
                kC, km = k @ C, k @ m                   # pre-update C and m (R1)
                G = gj * gj * G + gj * np.outer(k, kC)
                h = gj * gj * h + gj * k * km
                C = gj * C + np.outer(q, v)
                m = gj * m + q
                u = q @ S[b, j]
                o = u @ C - (q @ G if masked else 0.0)
                if normalize:
                    o = o / (u @ m - (q @ h if masked else 0.0) + eps)
                out[b, hh] = o
                hs["C"][b, hh], hs["G"][b, hh], hs["m"][b, hh], hs["h"][b, hh] = C, G, m, h
    return S, hs, out
