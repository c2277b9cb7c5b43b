"""Seeded synthetic workloads for masked second-order HLA.

This module draws random inputs and nothing else: it holds none of the method's
arithmetic, so both the CUDA path and the float64 oracle can be fed from it.

Every draw uses a torch generator (CPU unless a device is asked for) seeded per
workload (the tiny check uses seed 0, the others their index 2..5), draws q, k, v
(then dO) in float32 in that order, applies the workload's transform, and casts each
tensor to the workload dtype.
The oracle receives the cast values upcast to float32/float64, so both sides see
exactly the same numbers.

Workloads (sizes and distributions of the benchmark configurations):
  tiny      B=1 H=1  n=64    d=dv=16  fp32; q,k,v ~ N(0,1)/sqrt(d); decay 1; chunk 16
  normed    B=2 H=8  n=2048  d=dv=64  bf16; q,k = softplus(N(0,1)), v ~ N(0,1);
            ratio-normalised (eps 1e-6); decay linspace(0.95, 0.999, H); chunk 64
  long      B=1 H=16 n=65536 d=dv=64  bf16; q,k,v ~ N(0,1)/sqrt(d); unnormalised;
            decay linspace(0.99, 0.9999, H); chunk 128
  decode    256 sequences x H=32, d=dv=128; 4096-token bf16 prefill, N(0,1)/sqrt(d),
            decay 0.999; then single-token steps with fresh draws (seed 4000 + step)
  train     B=4 H=16 n=8192  d=dv=128 bf16; q,k,v ~ N(0,1)/sqrt(d); dO ~ N(0,1);
            decay 0.995; unnormalised; forward + backward; chunk 128
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    n: int
    d: int
    dv: int
    dtype: torch.dtype
    seed: int
    qk: str                 # "gauss" (N(0,1)/sqrt(d)) or "softplus" (softplus(N(0,1)))
    v_scale: str            # "gauss_sqrt_d" or "unit"
    gamma: tuple = field(default=None)   # (lo, hi) linspace over heads, or (g,) constant
    normalize: bool = False
    eps: float = 1e-6
    chunk: int = 64
    with_dout: bool = False

    @property
    def tokens(self) -> int:
        return self.B * self.H * self.n


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 64, 16, 16, torch.float32, 0, "gauss", "gauss_sqrt_d",
                     None, False, 1e-6, 16),
    "normed": Workload("normed", 2, 8, 2048, 64, 64, torch.bfloat16, 2, "softplus", "unit",
                       (0.95, 0.999), True, 1e-6, 64),
    "long": Workload("long", 1, 16, 65536, 64, 64, torch.bfloat16, 3, "gauss", "gauss_sqrt_d",
                     (0.99, 0.9999), False, 1e-6, 128),
    "decode_prefill": Workload("decode_prefill", 256, 32, 4096, 128, 128, torch.bfloat16, 4,
                               "gauss", "gauss_sqrt_d", (0.999,), False, 1e-6, 64),
    "train": Workload("train", 4, 16, 8192, 128, 128, torch.bfloat16, 5, "gauss",
                      "gauss_sqrt_d", (0.995,), False, 1e-6, 128, True),
}

DECODE_STEPS = 1024


def gammas(w: Workload) -> torch.Tensor | None:
    """Per-head decay values [H] float32 (None: no decay)."""
    if w.gamma is None:
        return None
    if len(w.gamma) == 1:
        return torch.full((w.H,), float(w.gamma[0]), dtype=torch.float32)
    lo, hi = w.gamma
    return torch.linspace(lo, hi, w.H, dtype=torch.float64).to(torch.float32)


def _draw_qkv(gen, B, H, n, d, dv, qk, v_scale, dtype=torch.float32):
    """q, k, v drawn in float32 in that order, transformed, then cast one at a time."""
    dev = gen.device

    def one(shape, kind, dim):
        x = torch.randn(shape, generator=gen, dtype=torch.float32, device=dev)
        if kind == "softplus":
            x = torch.nn.functional.softplus(x)
        elif kind in ("gauss", "gauss_sqrt_d"):
            x = x / math.sqrt(dim)
        return x.to(dtype)

    q = one((B, H, n, d), qk, d)
    k = one((B, H, n, d), qk, d)
    v = one((B, H, n, dv), v_scale, dv)
    return q, k, v


def make(w: Workload | str, n: int | None = None, B: int | None = None, H: int | None = None,
         seed: int | None = None, device="cpu"):
    """Draw a workload's inputs, cast to its dtype.

    ``n``, ``B``, ``H`` and ``seed`` override the workload's values to make smaller
    cases with the same distributions.  ``device`` selects the generator (a CUDA
    generator draws different numbers than the CPU one for the same seed; the oracle
    then receives copies of the drawn values).  Returns a dict with q, k, v (and dout),
    gamma [H] float32 (on the CPU) or None, and the workload flags.
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    B = w.B if B is None else B
    H = w.H if H is None else H
    n = w.n if n is None else n
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    q, k, v = _draw_qkv(gen, B, H, n, w.d, w.dv, w.qk, w.v_scale, dtype=w.dtype)
    out = {
        "q": q, "k": k, "v": v,
        "normalize": w.normalize, "eps": w.eps, "chunk": w.chunk,
    }
    if w.with_dout:
        out["dout"] = torch.randn((B, H, n, w.dv), generator=gen, dtype=torch.float32,
                                  device=device).to(w.dtype)
    g = gammas(w)
    if g is not None and H != w.H:
        g = torch.linspace(w.gamma[0], w.gamma[-1], H, dtype=torch.float64).to(torch.float32) \
            if len(w.gamma) == 2 else torch.full((H,), float(w.gamma[0]), dtype=torch.float32)
    out["gamma"] = g
    return out


def make_custom(B, H, n, d, dv, dtype=torch.bfloat16, seed=0, qk="gauss", v_scale="gauss_sqrt_d",
                gamma=None, with_dout=False):
    """Arbitrary-shape draw with the same recipe (edge cases and sweeps).

    ``gamma`` is None, a float, or a (lo, hi) pair for a linspace over heads.
    """
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    q, k, v = _draw_qkv(gen, B, H, n, d, dv, qk, v_scale, dtype=dtype)
    out = {"q": q, "k": k, "v": v}
    if with_dout:
        out["dout"] = torch.randn((B, H, n, dv), generator=gen, dtype=torch.float32).to(dtype)
    if gamma is None:
        out["gamma"] = None
    elif isinstance(gamma, (int, float)):
        out["gamma"] = torch.full((H,), float(gamma), dtype=torch.float32)
    else:
        out["gamma"] = torch.linspace(gamma[0], gamma[1], H, dtype=torch.float64).to(torch.float32)
    return out


def decode_step_inputs(step: int, N: int, H: int, d: int, dv: int, dtype=torch.bfloat16,
                       device="cpu"):
    """Fresh q, k, v [N, H, d|dv] for decode step ``step`` (seed 4000 + step),
    N(0,1)/sqrt(d) like the prefill.  Drawn on ``device``."""
    gen = torch.Generator(device=device)
    gen.manual_seed(4000 + step)
    q = torch.randn((N, H, d), generator=gen, device=device, dtype=torch.float32) / math.sqrt(d)
    k = torch.randn((N, H, d), generator=gen, device=device, dtype=torch.float32) / math.sqrt(d)
    v = torch.randn((N, H, dv), generator=gen, device=device, dtype=torch.float32) / math.sqrt(dv)
    return q.to(dtype), k.to(dtype), v.to(dtype)
