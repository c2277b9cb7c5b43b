"""GPU AHLA forward (chunk-parallel, mma.sync) against the float64 AHLA oracle, through the
C ABI.  Bar: max|gpu - oracle| / max|oracle| <= 2e-2 (bf16 inputs; the oracle runs on the
same bf16-rounded values)."""
import numpy as np
import pytest
import torch

import chunked_scan_mixer_gb300 as hla
from chunked_scan_mixer_gb300 import HLA2Error, inputs
from oracle import ahla_oracle as A

from .helpers import np32, np64, rel_err

pytestmark = pytest.mark.gpu


def run(x, chunk, normalize=False):
    g = None if x["gamma"] is None else x["gamma"].cuda()
    return hla.ahla_forward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), gamma=g, chunk=chunk,
                            normalize=normalize).cpu()


def oracle(x, normalize=False):
    g = None if x["gamma"] is None else x["gamma"].double().numpy()
    return A.serial_forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), g, normalize=normalize)


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("chunk", [32, 64])
def test_matches_oracle(d, chunk):
    x = inputs.make_custom(1, 3, 5 * chunk + 11, d, d, torch.bfloat16, seed=d + chunk, gamma=(0.9, 0.999))
    assert rel_err(np64(run(x, chunk)), oracle(x)) <= 2e-2


@pytest.mark.parametrize("n", [1, 17, 64, 300, 2049])
def test_lengths(n):
    x = inputs.make_custom(2, 2, n, 64, 64, torch.bfloat16, seed=n, gamma=(0.95, 0.9995))
    o = run(x, 64)
    assert torch.isfinite(o.float()).all()
    assert rel_err(np64(o), oracle(x)) <= 2e-2


@pytest.mark.parametrize("gamma", [None, 0.9, (0.5, 0.999)])
def test_decays(gamma):
    x = inputs.make_custom(2, 2, 700, 32, 32, torch.bfloat16, seed=7, gamma=gamma)
    assert rel_err(np64(run(x, 32)), oracle(x)) <= 2e-2


@pytest.mark.parametrize("d", [32, 64])
def test_normalized(d):
    """Positive q, k keep the denominator (the same cascade with v -> 1) away from zero."""
    x = inputs.make_custom(2, 2, 900, d, d, torch.bfloat16, seed=11 + d, qk="softplus", v_scale="unit",
                           gamma=(0.95, 0.999))
    assert rel_err(np64(run(x, 64, normalize=True)), oracle(x, normalize=True)) <= 2e-2


def test_many_segments_and_heads():
    """Many heads and several chunks per segment: exercises the carried state inside a CTA,
    the segment summaries (P, E, R) and the scan's cross term."""
    x = inputs.make_custom(2, 16, 128 * 40 + 5, 64, 64, torch.bfloat16, seed=12, gamma=(0.98, 0.9999))
    assert rel_err(np64(run(x, 64)), oracle(x)) <= 2e-2


def test_long_context_two_heads():
    """The long-context length (n = 65536, d = 64) on two heads of the decay range."""
    x = inputs.make_custom(1, 2, 65536, 64, 64, torch.bfloat16, seed=13, gamma=(0.99, 0.9999))
    assert rel_err(np64(run(x, 64)), oracle(x)) <= 2e-2


def test_causality_bit_exact():
    x = inputs.make_custom(1, 2, 1000, 64, 64, torch.bfloat16, seed=14, gamma=0.995)
    a = run(x, 64)
    y = {key: (t.clone() if isinstance(t, torch.Tensor) else t) for key, t in x.items()}
    for key in ("q", "k", "v"):
        y[key][:, :, 640:] = (y[key][:, :, 640:].float() * 2 + 1).to(torch.bfloat16)
    b = run(y, 64)
    assert torch.equal(a[:, :, :640], b[:, :, :640])


def test_rejects_uncovered_requests():
    x = inputs.make_custom(1, 1, 64, 64, 32, torch.bfloat16, seed=15)
    with pytest.raises(HLA2Error):  # d != dv
        hla.ahla_forward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), chunk=64)
    x = inputs.make_custom(1, 1, 64, 32, 32, torch.bfloat16, seed=15)
    with pytest.raises(HLA2Error):  # chunk 128 only for d = 64
        hla.ahla_forward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), chunk=128)


@pytest.mark.parametrize("n", [1, 127, 128, 129, 1000, 128 * 37 + 5])
def test_tcgen05_path_lengths(n):
    """chunk 128, d = dv = 64 runs the tcgen05 kernel."""
    x = inputs.make_custom(1, 3, n, 64, 64, torch.bfloat16, seed=20 + n % 97, gamma=(0.97, 0.9999))
    o = run(x, 128)
    assert torch.isfinite(o.float()).all()
    assert rel_err(np64(o), oracle(x)) <= 2e-2
    hla.check_status()


@pytest.mark.parametrize("gamma", [None, 0.9, (0.5, 0.999)])
def test_tcgen05_path_decays_and_mma_agreement(gamma):
    x = inputs.make_custom(2, 2, 1500, 64, 64, torch.bfloat16, seed=21, gamma=gamma)
    a, b = np64(run(x, 128)), np64(run(x, 64))
    ref = oracle(x)
    assert rel_err(a, ref) <= 2e-2 and rel_err(b, ref) <= 2e-2


def test_tcgen05_path_many_segments():
    """Several chunks per segment and many segments per head (summaries, scan, carries)."""
    x = inputs.make_custom(1, 16, 128 * 60 + 77, 64, 64, torch.bfloat16, seed=22, gamma=(0.98, 0.9999))
    assert rel_err(np64(run(x, 128)), oracle(x)) <= 2e-2
    hla.check_status()


def test_tcgen05_path_long_context_and_causality():
    x = inputs.make_custom(1, 2, 65536, 64, 64, torch.bfloat16, seed=23, gamma=(0.99, 0.9999))
    a = run(x, 128)
    assert rel_err(np64(a), oracle(x)) <= 2e-2
    y = {key: (t.clone() if isinstance(t, torch.Tensor) else t) for key, t in x.items()}
    for key in ("q", "k", "v"):
        y[key][:, :, 40000:] = (y[key][:, :, 40000:].float() * -1.5).to(torch.bfloat16)
    assert torch.equal(run(y, 128)[:, :, :40000], a[:, :, :40000])


def test_tcgen05_path_rejects_normalized():
    x = inputs.make_custom(1, 1, 64, 64, 64, torch.bfloat16, seed=24)
    with pytest.raises(HLA2Error):
        hla.ahla_forward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), chunk=128, normalize=True)


def _oracle_state_flat(st):
    B, H = st["P"].shape[:2]
    return np.concatenate([st["P"].reshape(B, H, -1), st["E"].reshape(B, H, -1), st["m"], st["n"]], axis=-1)


@pytest.mark.parametrize("chunk", [32, 64])
def test_final_state_matches_oracle(chunk):
    """The state after the last token (P | E | m | n) equals the oracle's serial state."""
    x = inputs.make_custom(2, 3, 777, 64, 64, torch.bfloat16, seed=30 + chunk, gamma=(0.95, 0.999))
    g = x["gamma"].cuda()
    o, fin = hla.ahla_forward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), gamma=g, chunk=chunk,
                              return_final_state=True)
    ref_o, st = A.serial_forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), x["gamma"].double().numpy(),
                                 return_state=True)
    assert rel_err(np64(o.cpu()), ref_o) <= 2e-2
    ref = _oracle_state_flat(st)
    got = fin.cpu().double().numpy()
    d = 64
    for lo, hi in ((0, d * d), (d * d, 2 * d * d), (2 * d * d, 2 * d * d + d), (2 * d * d + d, 2 * d * d + 2 * d)):
        assert rel_err(got[..., lo:hi], ref[..., lo:hi]) <= 2e-2


@pytest.mark.parametrize("d, dv", [(16, 16), (64, 64), (128, 128), (32, 64)])
@pytest.mark.parametrize("normalize", [False, True])
def test_decode_from_zero_equals_forward(d, dv, normalize):
    """fp32 decode steps from the empty state reproduce the serial AHLA outputs."""
    N, H, n = 2, 3, 23
    x = inputs.make_custom(N, H, n, d, dv, torch.float32, seed=d + dv, qk="softplus" if normalize else "gauss",
                           gamma=(0.9, 0.99))
    state = torch.zeros((N, H, hla.ahla_state_floats(d, dv)), device="cuda")
    outs = [hla.ahla_decode_step(state, x["q"][:, :, t].cuda(), x["k"][:, :, t].cuda(), x["v"][:, :, t].cuda(),
                                 gamma=x["gamma"].cuda(), normalize=normalize, eps=1e-6) for t in range(n)]
    o = torch.stack(outs, dim=2).cpu()
    ref, st = A.serial_forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), x["gamma"].double().numpy(),
                               normalize=normalize, eps=1e-6, return_state=True)
    assert rel_err(np64(o), ref) <= 1e-4
    assert rel_err(state.cpu().double().numpy(), _oracle_state_flat(st)) <= 1e-5


def test_prefill_then_decode_matches_uninterrupted_oracle():
    """A GPU prefill's final state continues like the oracle run over prefill + decode tokens."""
    N, H, d, n, extra = 2, 4, 64, 500, 6
    x = inputs.make_custom(N, H, n + extra, d, d, torch.bfloat16, seed=31, gamma=0.995)
    g = x["gamma"].cuda()
    _, fin = hla.ahla_forward(x["q"][:, :, :n].contiguous().cuda(), x["k"][:, :, :n].contiguous().cuda(),
                              x["v"][:, :, :n].contiguous().cuda(), gamma=g, chunk=64, return_final_state=True)
    ref = A.serial_forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), x["gamma"].double().numpy())
    for t in range(n, n + extra):
        o = hla.ahla_decode_step(fin, x["q"][:, :, t].cuda(), x["k"][:, :, t].cuda(), x["v"][:, :, t].cuda(), gamma=g)
        assert rel_err(np64(o.cpu()), ref[:, :, t]) <= 2e-2, t


def test_final_state_at_chunk_128_runs_at_width_64():
    """The tcgen05 AHLA kernel keeps no final state, so a chunk-128 call that asks for one runs
    at width 64: the same output and state, bit for bit, as the chunk-64 call, the state against
    the oracle's, and the workspace query at chunk 128 covers it."""
    N, H, d, n = 2, 4, 64, 700
    x = inputs.make_custom(N, H, n, d, d, torch.bfloat16, seed=32, gamma=(0.99, 0.999))
    g = x["gamma"].cuda()
    args = (x["q"].cuda(), x["k"].cuda(), x["v"].cuda())
    o128, f128 = hla.ahla_forward(*args, gamma=g, chunk=128, return_final_state=True)
    o64, f64 = hla.ahla_forward(*args, gamma=g, chunk=64, return_final_state=True)
    assert torch.equal(o128, o64) and torch.equal(f128, f64)
    L = hla.lib()
    assert L.hla2_ahla_forward_workspace_bytes(N, H, n, d, d, 128, 1, 0) >= \
        L.hla2_ahla_forward_workspace_bytes(N, H, n, d, d, 64, 1, 0)
    _, st = A.serial_forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), x["gamma"].double().numpy(), return_state=True)
    assert rel_err(f128.cpu().double().numpy(), _oracle_state_flat(st)) <= 2e-2


@pytest.mark.parametrize("chunk", [32, 64, 128])
@pytest.mark.parametrize("normalize", [False, True])
def test_continuation_from_init_state(chunk, normalize):
    """A forward over [m, n) from the GPU state after [0, m) equals the oracle run over all
    of [0, n), on every AHLA kernel (chunk 128 is the tcgen05 one)."""
    if normalize and chunk == 128:
        pytest.skip("the tcgen05 kernel is unnormalised")
    N, H, d, n, m = 2, 4, 64, 900, 333
    x = inputs.make_custom(N, H, n, d, d, torch.bfloat16, seed=33 + chunk, gamma=(0.99, 0.999),
                           qk="softplus" if normalize else "gauss", v_scale="unit" if normalize else "gauss_sqrt_d")
    g = x["gamma"].cuda()
    q, k, v = (x[key].cuda() for key in ("q", "k", "v"))
    _, fin = hla.ahla_forward(q[:, :, :m].contiguous(), k[:, :, :m].contiguous(), v[:, :, :m].contiguous(), gamma=g,
                              chunk=64, normalize=normalize, return_final_state=True)
    o2 = hla.ahla_forward(q[:, :, m:].contiguous(), k[:, :, m:].contiguous(), v[:, :, m:].contiguous(), gamma=g,
                          chunk=chunk, normalize=normalize, init_state=fin)
    ref = A.serial_forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), x["gamma"].double().numpy(), normalize=normalize)
    assert rel_err(np64(o2.cpu()), ref[:, :, m:]) <= 2e-2


def test_empty_sequence_passes_init_state_through():
    x = inputs.make_custom(1, 2, 0, 32, 32, torch.bfloat16, seed=34)
    init = torch.randn(1, 2, hla.ahla_state_floats(32, 32), device="cuda")
    _, fin = hla.ahla_forward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), chunk=32, init_state=init,
                              return_final_state=True)
    assert torch.equal(fin, init)


# ---- reverse mode ------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("d, chunk, n", [(16, 16, 77), (32, 32, 300), (64, 32, 500), (128, 16, 90), (64, 64, 1000)])
def test_backward_matches_the_oracle_adjoint(dtype, d, chunk, n):
    """AHLA gradients against the oracle's reverse sweep of the serial recurrence, across
    chunks, segments and a ragged tail."""
    x = inputs.make_custom(1, 2, n, d, d, dtype, seed=d + chunk + n, gamma=(0.95, 0.999), with_dout=True)
    got = hla.ahla_backward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["dout"].cuda(), gamma=x["gamma"].cuda(),
                            chunk=chunk)
    ref = A.serial_backward(np32(x["q"]), np32(x["k"]), np32(x["v"]), np32(x["dout"]), x["gamma"].double().numpy())
    tol = 1e-4 if dtype == torch.float32 else 2e-2
    for name, gg, rr in zip(("dq", "dk", "dv"), got, ref):
        assert rel_err(np64(gg.cpu()), rr) <= tol, name


def test_backward_tiny_against_the_pair_sum_gradients():
    x = inputs.make_custom(1, 1, 20, 16, 16, torch.float32, seed=99, gamma=0.9, with_dout=True)
    got = hla.ahla_backward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["dout"].cuda(), gamma=x["gamma"].cuda(),
                            chunk=16)
    ref = A.pairsum_grads(np32(x["q"]), np32(x["k"]), np32(x["v"]), np32(x["dout"]), [0.9])
    for name, gg, rr in zip(("dq", "dk", "dv"), got, ref):
        assert rel_err(np64(gg.cpu()), rr) <= 1e-4, name


def test_backward_many_segments_no_decay():
    x = inputs.make_custom(2, 2, 2500, 32, 32, torch.float32, seed=98, gamma=None, with_dout=True)
    got = hla.ahla_backward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["dout"].cuda(), chunk=16)
    ref = A.serial_backward(np32(x["q"]), np32(x["k"]), np32(x["v"]), np32(x["dout"]), None)
    for name, gg, rr in zip(("dq", "dk", "dv"), got, ref):
        assert rel_err(np64(gg.cpu()), rr) <= 1e-4, name
