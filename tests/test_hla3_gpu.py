"""GPU masked third-order output (gamma = 1) against the float64 oracle
(``oracle/hla3_oracle.py``), through the C ABI.  Bars: 1e-4 for float32 inputs, 2e-2 for
bf16 inputs (the oracle runs on the same bf16-rounded values)."""
import ctypes

import numpy as np
import pytest
import torch

import chunked_scan_mixer_gb300 as hla
from chunked_scan_mixer_gb300 import inputs
from chunked_scan_mixer_gb300.hla2 import Opts
from oracle import hla3_oracle as O3

from .helpers import np64, rel_err, tol_for

pytestmark = pytest.mark.gpu


def run(x, **kw):
    return hla.hla3_forward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), **kw).cpu()


def test_tiny_fp32_against_the_triple_sum():
    x = inputs.make_custom(1, 2, 24, 16, 16, torch.float32, seed=80)
    ref = O3.brute_force_forward(np64(x["q"]), np64(x["k"]), np64(x["v"]))
    for chunk in (16, 32):
        assert rel_err(np64(run(x, chunk=chunk)), ref) <= 1e-4, chunk


@pytest.mark.parametrize("d, dv, chunk, n", [(32, 64, 16, 300), (64, 32, 32, 333), (16, 128, 64, 200),
                                              (128, 128, 32, 150)])
def test_fp32_shapes_and_segments(d, dv, chunk, n):
    x = inputs.make_custom(1, 2, n, d, dv, torch.float32, seed=d + dv + n)
    ref = O3.serial_forward(np64(x["q"]), np64(x["k"]), np64(x["v"]))
    assert rel_err(np64(run(x, chunk=chunk)), ref) <= 1e-4


@pytest.mark.parametrize("chunk, n", [(64, 1000), (128, 1000), (128, 129), (32, 77)])
def test_bf16(chunk, n):
    """chunk 128 at d = 64 runs the second pass on the tcgen05 kernels."""
    x = inputs.make_custom(1, 3, n, 64, 64, torch.bfloat16, seed=81 + n)
    ref = O3.serial_forward(np64(x["q"]), np64(x["k"]), np64(x["v"]))
    assert rel_err(np64(run(x, chunk=chunk)), ref) <= 2e-2


def test_bf16_segments_of_several_chunks():
    """24 heads of 2048 tokens: the first-order pass runs 6 segments of 3 chunks per head, so
    its summary and output pipelines reuse their stages within a segment."""
    x = inputs.make_custom(1, 24, 2048, 64, 64, torch.bfloat16, seed=85)
    ref = O3.serial_forward(np64(x["q"]), np64(x["k"]), np64(x["v"]))
    assert rel_err(np64(run(x, chunk=128)), ref) <= 2e-2


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_normalized(dtype):
    x = inputs.make_custom(2, 2, 260, 32, 32, dtype, seed=82, qk="softplus", v_scale="unit")
    ref = O3.serial_forward(np64(x["q"]), np64(x["k"]), np64(x["v"]), normalize=True, eps=1e-6)
    got = run(x, chunk=32, normalize=True, eps=1e-6)
    assert rel_err(np64(got), ref) <= tol_for(dtype)


def test_causality():
    x = inputs.make_custom(1, 2, 300, 32, 32, torch.float32, seed=83)
    a = run(x, chunk=32)
    y = {key: (val.clone() if key in ("q", "k", "v") else val) for key, val in x.items()}
    y["q"][:, :, 200:] += 1.0
    y["v"][:, :, 200:] = 0
    b = run(y, chunk=32)
    assert torch.equal(a[:, :, :200], b[:, :, :200])


def test_decay_is_refused():
    L = hla.lib()
    p = ctypes.c_void_p(16)
    g = torch.full((1,), 0.9, device="cuda")
    o = Opts(0, 1e-6, None, 0, None, None, None, 0, 0)
    rc = L.hla2_hla3_forward(p, p, p, p, 1, 1, 16, 16, 16, ctypes.c_void_p(g.data_ptr()), 0, 16, None,
                             ctypes.byref(o))
    assert rc == -2 and b"gamma" in L.hla2_last_error()
    assert np.isfinite(rc)


def test_bf16_first_order_paths_agree():
    """bf16 d = dv = 64 without a final state runs the first-order pass on the d = 64 first-order
    scan kernels (with a final state: the AHLA tcgen05 kernel in its first-order mode, covered by
    the prefill tests below); with the tcgen05 kernels disabled it runs on the SIMT kernel.  Both
    against the oracle, several segments."""
    import os

    x = inputs.make_custom(2, 4, 128 * 30 + 7, 64, 64, torch.bfloat16, seed=84)
    ref = O3.serial_forward(np64(x["q"]), np64(x["k"]), np64(x["v"]))
    a = run(x, chunk=128)
    old = os.environ.get("HLA2_KERNEL")
    os.environ["HLA2_KERNEL"] = "mma"
    try:
        b = run(x, chunk=128)
    finally:
        if old is None:
            os.environ.pop("HLA2_KERNEL", None)
        else:
            os.environ["HLA2_KERNEL"] = old
    hla.check_status()
    assert rel_err(np64(a), ref) <= 2e-2
    assert rel_err(np64(b), ref) <= 2e-2


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("d, dv", [(16, 16), (64, 64), (128, 128), (32, 64)])
@pytest.mark.parametrize("normalize", [False, True])
def test_decode_from_zero_equals_forward(dtype, d, dv, normalize):
    """Streaming steps from the empty state reproduce the oracle's outputs token by token,
    and agree with the chunked GPU forward on the same tokens."""
    N, H, n = 2, 3, 21
    x = inputs.make_custom(N, H, n, d, dv, dtype, seed=d + dv + 90, qk="softplus" if normalize else "gauss",
                           v_scale="unit" if normalize else "gauss_sqrt_d")
    state = torch.zeros((N, H, O3.state_floats(d, dv)), device="cuda")
    outs = [hla.hla3_decode_step(state, x["q"][:, :, t].cuda(), x["k"][:, :, t].cuda(), x["v"][:, :, t].cuda(),
                                 normalize=normalize, eps=1e-6) for t in range(n)]
    o = torch.stack(outs, dim=2).cpu()
    ref = O3.serial_forward(np64(x["q"]), np64(x["k"]), np64(x["v"]), normalize=normalize, eps=1e-6)
    assert rel_err(np64(o), ref) <= tol_for(dtype)
    fwd = run(x, chunk=16, normalize=normalize, eps=1e-6)
    assert rel_err(np64(fwd), ref) <= tol_for(dtype)
    # and the state after the last step is the oracle's
    st = np.zeros((N, H, O3.state_floats(d, dv)))
    for t in range(n):
        O3.decode_step(st, np64(x["q"][:, :, t]), np64(x["k"][:, :, t]), np64(x["v"][:, :, t]), normalize)
    assert rel_err(state.cpu().double().numpy(), st) <= 1e-5


@pytest.mark.parametrize("dtype, d, chunk", [(torch.float32, 32, 32), (torch.bfloat16, 64, 128), (torch.bfloat16, 32, 64)])
@pytest.mark.parametrize("normalize", [False, True])
def test_prefill_then_decode_matches_the_oracle(dtype, d, chunk, normalize):
    """The forward's final state (prefill) equals the oracle's streaming state, and decode steps
    continued from it reproduce the oracle's outputs over prefill + decode tokens."""
    N, H, n0, steps = 2, 3, 200, 5
    x = inputs.make_custom(N, H, n0 + steps, d, d, dtype, seed=d + chunk + 95, qk="softplus" if normalize else "gauss",
                           v_scale="unit" if normalize else "gauss_sqrt_d")
    q, k, v = (x[key].cuda() for key in ("q", "k", "v"))
    _, state = hla.hla3_forward(q[:, :, :n0].contiguous(), k[:, :, :n0].contiguous(), v[:, :, :n0].contiguous(),
                                chunk=chunk, normalize=normalize, eps=1e-6, return_final_state=True)
    st = np.zeros((N, H, O3.state_floats(d, d)))
    for t in range(n0):
        O3.decode_step(st, np64(x["q"][:, :, t]), np64(x["k"][:, :, t]), np64(x["v"][:, :, t]), normalize)
    tol_state = 1e-4 if dtype == torch.float32 else 2e-2
    got = state.cpu().double().numpy()
    sizes = (d * d, d * d, d * d, d, d)  # S, P, Y, m, y
    off = 0
    for name, size in zip(("S", "P", "Y", "m", "y"), sizes):
        assert rel_err(got[..., off:off + size], st[..., off:off + size]) <= tol_state, name
        off += size
    ref = O3.serial_forward(np64(x["q"]), np64(x["k"]), np64(x["v"]), normalize=normalize, eps=1e-6)
    for t in range(n0, n0 + steps):
        o = hla.hla3_decode_step(state, q[:, :, t], k[:, :, t], v[:, :, t], normalize=normalize, eps=1e-6)
        assert rel_err(np64(o.cpu()), ref[:, :, t]) <= tol_for(dtype), t
