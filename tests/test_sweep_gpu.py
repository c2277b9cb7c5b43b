"""Seeded random sweep of the public forward and backward calls against the float64 oracle.

The targeted tests enumerate one or two factors at a time; here each case draws all of them
at once (dtype, d, dv, chunk width, batch and heads, length exact or ragged, decay none,
scalar or per head, masked or unmasked output, ratio normalisation, a carried-in state and
a returned final state), so that combinations no single test names are exercised too.
Every case is fixed by its index: a failure names the case, and the case rebuilds from it.

Bars as everywhere: max|gpu - oracle| / max|oracle| <= 1e-4 for float32 inputs and
<= 2e-2 for bf16 inputs, per output and per part of the state."""
import random

import numpy as np
import pytest
import torch

import chunked_scan_mixer_gb300 as hla
from chunked_scan_mixer_gb300 import HLA2Error, inputs
from oracle import cref
from oracle import hla2_oracle as O

from .helpers import np32, np64, rel_err, tol_for

pytestmark = pytest.mark.gpu

DIMS = (16, 32, 64, 128)
CHUNKS = (16, 32, 64, 128)
MAX_TOKENS = 24000  # B * H * n per case, so that the serial oracle stays well under a second


def _length(rng, chunk):
    kind = rng.randrange(6)
    if kind == 0:
        return rng.choice((1, 2, chunk - 1, chunk, chunk + 1))
    if kind == 1:
        return chunk * rng.randint(2, 24)                  # whole chunks
    if kind == 2:
        return chunk * rng.randint(2, 24) + rng.choice((1, chunk - 1))
    return rng.randint(3, 3000)


def _gamma(rng):
    kind = rng.randrange(3)
    if kind == 0:
        return None
    if kind == 1:
        return rng.uniform(0.9, 1.0)
    lo = rng.uniform(0.8, 0.999)
    return (lo, rng.uniform(lo, 1.0))


def forward_case(i):
    rng = random.Random(1000 + i)
    dtype = torch.bfloat16 if rng.random() < 0.65 else torch.float32
    if dtype == torch.bfloat16 and rng.random() < 0.4:
        d = dv = 64                                         # the tensor-core shapes
        chunk = rng.choice((64, 128, 128))
    else:
        d = rng.choice(DIMS)
        dv = d if rng.random() < 0.6 else rng.choice(DIMS)
        chunk = rng.choice(CHUNKS)
    B = rng.choice((1, 1, 2))
    H = rng.choice((1, 2, 3, 5, 16))
    n = _length(rng, chunk)
    n = max(1, min(n, MAX_TOKENS // (B * H)))
    masked = rng.random() < 0.75
    normalize = rng.random() < 0.25
    return dict(dtype=dtype, d=d, dv=dv, chunk=chunk, B=B, H=H, n=n, masked=masked, normalize=normalize,
                gamma=_gamma(rng), init=rng.random() < 0.3, final=rng.random() < 0.4, seed=7000 + i,
                prefix=rng.randint(1, 300))


def _draw(c, n, seed):
    if c["normalize"]:  # positive queries and keys keep the denominator away from zero
        return inputs.make_custom(c["B"], c["H"], n, c["d"], c["dv"], c["dtype"], seed=seed, qk="softplus",
                                  v_scale="unit", gamma=c["gamma"])
    return inputs.make_custom(c["B"], c["H"], n, c["d"], c["dv"], c["dtype"], seed=seed, gamma=c["gamma"])


@pytest.mark.parametrize("i", range(48))
def test_forward_sweep(i):
    c = forward_case(i)
    x = _draw(c, c["n"], c["seed"])
    g64 = None if x["gamma"] is None else x["gamma"].double().numpy()
    init = None
    if c["init"]:
        # a state that real tokens reach: the oracle's final state after a prefix of the same kind
        pre = _draw(c, c["prefix"], c["seed"] + 1)
        _, init = cref.forward(np32(pre["q"]), np32(pre["k"]), np32(pre["v"]), g64, return_state=True)
        if not c["masked"]:  # the unmasked output keeps no G and h
            parts = O.unpack_state(init, c["d"], c["dv"])  # views into init
            parts["G"][...] = 0.0
            parts["h"][...] = 0.0
        init = init.astype(np.float32)
    ref = cref.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), g64, normalize=c["normalize"], eps=1e-6,
                       init_state=None if init is None else init.astype(np.float64),
                       return_state=c["final"], masked=c["masked"])
    ref_o, ref_state = ref if c["final"] else (ref, None)
    try:
        res = hla.forward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(),
                          gamma=None if x["gamma"] is None else x["gamma"].cuda(), normalize=c["normalize"],
                          chunk=c["chunk"], eps=1e-6, init_state=None if init is None else torch.from_numpy(init).cuda(),
                          return_final_state=c["final"], masked=c["masked"])
    except HLA2Error as e:
        if e.code == -2:  # a request outside the compiled kernel set is reported, not run
            pytest.skip(str(e))
        raise
    hla.check_status()
    o, fin = res if c["final"] else (res, None)
    tol = tol_for(c["dtype"])
    assert o.shape == (c["B"], c["H"], c["n"], c["dv"]) and o.dtype == c["dtype"]
    assert torch.isfinite(o.float()).all(), c
    assert rel_err(np64(o.cpu()), ref_o) <= tol, c
    if c["final"]:
        got = O.unpack_state(np64(fin.cpu()), c["d"], c["dv"])
        want = O.unpack_state(ref_state, c["d"], c["dv"])
        for key in ("S", "C", "m", "G", "h") if c["masked"] else ("S", "C", "m"):
            assert rel_err(got[key], want[key]) <= tol, (key, c)
        if not c["masked"]:
            assert not got["G"].any() and not got["h"].any(), c


def backward_case(i):
    rng = random.Random(2000 + i)
    dtype = torch.bfloat16 if rng.random() < 0.6 else torch.float32
    d = rng.choice(DIMS)
    dv = d if dtype == torch.bfloat16 or rng.random() < 0.5 else rng.choice(DIMS)
    chunk = rng.choice(CHUNKS)  # the backward runs at the widest width <= chunk with a kernel
    B, H = rng.choice((1, 2)), rng.choice((1, 2, 3))
    n = max(1, min(_length(rng, chunk), 8000 // (B * H)))
    normalize = rng.random() < 0.3
    if normalize:
        # One token alone: the ratio-normalised output is v (q.k)^2 / ((q.k)^2 + eps), which
        # depends on q and k only through eps.  Its dq and dk are eps-sized differences of the
        # two quotient-rule terms (about 1e-8 of either), below float32 resolution, so the
        # relative bar has no meaning there; from two tokens on they are 5e-2 or more of them.
        n = max(n, 2)
    return dict(dtype=dtype, d=d, dv=dv, chunk=chunk, B=B, H=H, n=n, normalize=normalize,
                gamma=_gamma(rng), seed=9000 + i)


@pytest.mark.parametrize("i", range(20))
def test_backward_sweep(i):
    c = backward_case(i)
    kw = dict(qk="softplus", v_scale="unit") if c["normalize"] else {}
    x = inputs.make_custom(c["B"], c["H"], c["n"], c["d"], c["dv"], c["dtype"], seed=c["seed"], gamma=c["gamma"],
                           with_dout=True, **kw)
    g64 = None if x["gamma"] is None else x["gamma"].double().numpy()
    if c["normalize"]:
        ref = cref.backward_normalized(np32(x["q"]), np32(x["k"]), np32(x["v"]), np32(x["dout"]), g64, eps=1e-6)
    else:
        ref = cref.backward(np32(x["q"]), np32(x["k"]), np32(x["v"]), np32(x["dout"]), g64)
    try:
        got = hla.backward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["dout"].cuda(),
                           gamma=None if x["gamma"] is None else x["gamma"].cuda(), chunk=c["chunk"],
                           normalize=c["normalize"], eps=1e-6)
    except HLA2Error as e:
        if e.code == -2:
            pytest.skip(str(e))
        raise
    hla.check_status()
    for name, gg, rr in zip(("dq", "dk", "dv"), got, ref):
        assert torch.isfinite(gg.float()).all(), (name, c)
        assert rel_err(np64(gg.cpu()), rr) <= tol_for(c["dtype"]), (name, c)


def ahla_case(i):
    rng = random.Random(3000 + i)
    d = rng.choice(DIMS)
    normalize = rng.random() < 0.3
    final = rng.random() < 0.4
    tc_ok = d == 64 and not normalize and not final  # the tcgen05 AHLA kernel (chunk 128)
    chunk = rng.choice((32, 64, 128, 128) if tc_ok else (32, 64))
    B, H = rng.choice((1, 2)), rng.choice((1, 2, 3, 16))
    n = max(1, min(_length(rng, chunk), 12000 // (B * H)))
    return dict(d=d, chunk=chunk, B=B, H=H, n=n, normalize=normalize, final=final, gamma=_gamma(rng),
                prefix=rng.choice((0, 0, rng.randint(1, 200))), seed=11000 + i)


def _ahla_state_flat(st):
    B, H = st["P"].shape[:2]
    return np.concatenate([st["P"].reshape(B, H, -1), st["E"].reshape(B, H, -1), st["m"], st["n"]], axis=-1)


@pytest.mark.parametrize("i", range(24))
def test_ahla_forward_sweep(i):
    """The AHLA forward (bf16, d == dv) with the same kind of draws; a carried-in state comes
    from a GPU prefix call (chunk 64) and the oracle runs over prefix and sequence together."""
    from oracle import ahla_oracle as A

    c = ahla_case(i)
    d, m = c["d"], c["prefix"]
    kw = dict(qk="softplus", v_scale="unit") if c["normalize"] else {}
    x = inputs.make_custom(c["B"], c["H"], m + c["n"], d, d, torch.bfloat16, seed=c["seed"], gamma=c["gamma"], **kw)
    g = None if x["gamma"] is None else x["gamma"].cuda()
    q, k, v = (x[key].cuda() for key in ("q", "k", "v"))
    init = None
    if m:
        _, init = hla.ahla_forward(q[:, :, :m].contiguous(), k[:, :, :m].contiguous(), v[:, :, :m].contiguous(),
                                   gamma=g, chunk=64, normalize=c["normalize"], return_final_state=True)
    res = hla.ahla_forward(q[:, :, m:].contiguous(), k[:, :, m:].contiguous(), v[:, :, m:].contiguous(), gamma=g,
                           chunk=c["chunk"], normalize=c["normalize"], init_state=init,
                           return_final_state=c["final"])
    hla.check_status()
    o, fin = res if c["final"] else (res, None)
    g64 = None if x["gamma"] is None else x["gamma"].double().numpy()
    ref_o, st = A.serial_forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), g64, normalize=c["normalize"],
                                 return_state=True)
    assert torch.isfinite(o.float()).all(), c
    assert rel_err(np64(o.cpu()), ref_o[:, :, m:]) <= 2e-2, c
    if c["final"]:
        got, ref = np64(fin.cpu()), _ahla_state_flat(st)
        for lo, hi in ((0, d * d), (d * d, 2 * d * d), (2 * d * d, 2 * d * d + d), (2 * d * d + d, 2 * d * d + 2 * d)):
            assert rel_err(got[..., lo:hi], ref[..., lo:hi]) <= 2e-2, (lo, c)
