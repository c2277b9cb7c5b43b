"""Exact rational evaluation of the masked second-order HLA output (test infrastructure).

The plain definition of the strictly causal output, written with Python
``fractions.Fraction`` so that it carries no rounding at all:

    o_t   = sum_{j <= t} sum_{i <= j} g^((t-i)+(t-j)) (q_t . k_i)(k_i . q_j) v_j
    den_t = the same sum with v_j replaced by 1

(page "Higher-order Linear Attention", technical summary, item "1. Zweite Ordnung HLA":
the product q_t^T S_t C_t with the future terms removed; section summary §2.1: the
causal mask keeps positions on and before the current one; §4.3: fixed decay).
Used only to write the exact fixtures under ``tests/golden/``.
"""
from __future__ import annotations

from fractions import Fraction


def _dot(a, b):
    return sum((x * y for x, y in zip(a, b)), Fraction(0))


def pair_sum(q, k, v, g):
    """q, k: lists of n vectors (length d) of Fractions; v: n vectors (length dv);
    g: Fraction decay.  Returns (o, den): o a list of n vectors, den a list of n values."""
    n = len(q)
    dv = len(v[0]) if n else 0
    outs, dens = [], []
    for t in range(n):
        num = [Fraction(0)] * dv
        den = Fraction(0)
        for j in range(t + 1):
            w = Fraction(0)
            for i in range(j + 1):
                w += g ** ((t - i) + (t - j)) * _dot(q[t], k[i]) * _dot(k[i], q[j])
            num = [a + w * b for a, b in zip(num, v[j])]
            den += w
        outs.append(num)
        dens.append(den)
    return outs, dens
