"""GPU forward against the float64 oracle, through the C ABI.

Bars: max|gpu - oracle| / max|oracle| <= 1e-4 for float32 inputs and <= 2e-2 for
bf16 inputs (the oracle runs on the same bf16-rounded values)."""
import numpy as np
import pytest
import torch

import chunked_scan_mixer_gb300 as hla
from chunked_scan_mixer_gb300 import inputs
from oracle import cref
from oracle import hla2_oracle as O

from .helpers import np32, np64, rel_err, tol_for

pytestmark = pytest.mark.gpu


def run_gpu(x, **kw):
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    return hla.forward(q, k, v, gamma=None if x["gamma"] is None else x["gamma"].cuda(), **kw)


def oracle(x, normalize=False, eps=1e-6, init_state=None, return_state=False):
    g = None if x["gamma"] is None else x["gamma"].double().numpy()
    return cref.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), g, normalize=normalize, eps=eps,
                        init_state=init_state, return_state=return_state)


# ---- the benchmark workloads -------------------------------------------------------------

def test_tiny_fp32_against_brute_force_and_serial():
    x = inputs.make("tiny")
    o = run_gpu(x, chunk=16).cpu()
    ref = O.brute_force_forward(np64(x["q"]), np64(x["k"]), np64(x["v"]), None)
    assert rel_err(np64(o), ref) <= 1e-4
    assert rel_err(np64(o), oracle(x)) <= 1e-4


def test_normed_bf16_workload():
    x = inputs.make("normed")
    o = run_gpu(x, chunk=64, normalize=True, eps=x["eps"]).cpu()
    ref = oracle(x, normalize=True, eps=x["eps"])
    assert np.all(np.isfinite(np64(o)))
    assert rel_err(np64(o), ref) <= 2e-2


def test_mma_forward_is_reproducible():
    """The mma.sync forward adds the per-tile partial sums of the denominator rows and of the
    y moment in a fixed order: two runs of the normalised workload, and two runs of a call
    whose final state reads the y moment, give the same bits."""
    x = inputs.make("normed")
    a = run_gpu(x, chunk=64, normalize=True, eps=x["eps"])
    b = run_gpu(x, chunk=64, normalize=True, eps=x["eps"])
    assert torch.equal(a, b)
    y = inputs.make_custom(2, 4, 700, 64, 64, torch.bfloat16, seed=21, gamma=(0.97, 0.999))
    o1, s1 = run_gpu(y, chunk=64, return_final_state=True)
    o2, s2 = run_gpu(y, chunk=64, return_final_state=True)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    ref, ref_state = oracle(y, return_state=True)
    assert rel_err(np64(o1.cpu()), ref) <= 2e-2
    got, want = O.unpack_state(np64(s1.cpu()), 64, 64), O.unpack_state(ref_state, 64, 64)
    for key in ("S", "C", "m", "G", "h"):
        assert rel_err(got[key], want[key]) <= 2e-2, key


def test_long_context_full_size():
    """n = 65536, 16 heads, d = dv = 64: the benchmarked launch, every output compared."""
    x = inputs.make("long")
    o = run_gpu(x, chunk=x["chunk"]).cpu()
    ref = oracle(x)
    err = rel_err(np64(o), ref)
    assert err <= 2e-2, err
    # and per head (no head may hide behind a larger one)
    for h in range(16):
        assert rel_err(np64(o[0, h]), ref[0, h]) <= 2e-2


# ---- shapes, chunk widths, ragged lengths --------------------------------------------------

@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("chunk", [16, 32, 64, 128])
def test_bf16_shapes_and_chunks(d, chunk):
    # d = 128 at chunk 128 has no kernel (its tiles exceed one CTA's shared memory) and runs
    # at the widest narrower width that has one
    n = 3 * chunk + 5  # several chunks and a ragged tail
    x = inputs.make_custom(2, 3, n, d, d, torch.bfloat16, seed=d + chunk, gamma=(0.9, 1.0))
    o = run_gpu(x, chunk=chunk).cpu()
    assert rel_err(np64(o), oracle(x)) <= 2e-2


@pytest.mark.parametrize("d, dv", [(16, 16), (32, 32), (64, 64), (32, 64), (64, 16)])
@pytest.mark.parametrize("chunk", [16, 32])
def test_fp32_shapes(d, dv, chunk):
    n = 4 * chunk + 3
    x = inputs.make_custom(1, 2, n, d, dv, torch.float32, seed=7 * d + dv, gamma=(0.95, 0.999))
    o = run_gpu(x, chunk=chunk).cpu()
    assert rel_err(np64(o), oracle(x)) <= 1e-4


def test_bf16_unequal_dims_use_simt_path():
    x = inputs.make_custom(1, 2, 200, 32, 64, torch.bfloat16, seed=3, gamma=0.97)
    o = run_gpu(x, chunk=32).cpu()
    assert rel_err(np64(o), oracle(x)) <= 2e-2


@pytest.mark.parametrize("n", [1, 2, 15, 16, 17, 63, 64, 65, 1000])
def test_ragged_and_short_sequences(n):
    x = inputs.make_custom(1, 2, n, 64, 64, torch.bfloat16, seed=n, gamma=(0.9, 0.99))
    o = run_gpu(x, chunk=64).cpu()
    assert rel_err(np64(o), oracle(x)) <= 2e-2


def test_many_segments_long_sequence_fp32():
    """fp32 path across many segments: the inter-segment scan at 1e-4."""
    x = inputs.make_custom(1, 1, 4096, 16, 16, torch.float32, seed=11, gamma=0.999)
    o = run_gpu(x, chunk=16).cpu()
    assert rel_err(np64(o), oracle(x)) <= 1e-4


def test_no_decay_long_fp32():
    x = inputs.make_custom(1, 2, 1500, 16, 16, torch.float32, seed=12, gamma=None)
    o = run_gpu(x, chunk=32).cpu()
    assert rel_err(np64(o), oracle(x)) <= 1e-4


def test_chunk_width_independence_on_gpu():
    x = inputs.make_custom(1, 4, 777, 64, 64, torch.bfloat16, seed=13, gamma=(0.98, 0.9999))
    outs = [np64(run_gpu(x, chunk=c).cpu()) for c in (16, 32, 64, 128)]
    ref = oracle(x)
    for o in outs:
        assert rel_err(o, ref) <= 2e-2
    for o in outs[1:]:
        assert rel_err(o, outs[0]) <= 2e-2


@pytest.mark.parametrize("dtype, d, dv", [(torch.bfloat16, 128, 128), (torch.bfloat16, 128, 32),
                                           (torch.float32, 128, 128), (torch.float32, 64, 64)])
def test_chunk_wider_than_the_kernels_runs_narrower(dtype, d, dv, monkeypatch):
    """A chunk width with no chunk kernel for these sizes runs at the widest narrower width
    that has one: the same plan, workspace and output, bit for bit, as asking for that width.
    (bf16 at d = dv = 128 and chunk 128 otherwise runs on the first-order scans, so the chunk
    kernels are selected for it here.)"""
    if dtype == torch.bfloat16 and d == 128 and dv == 128:
        monkeypatch.setenv("HLA2_KERNEL", "mma")
    x = inputs.make_custom(1, 3, 1000, d, dv, dtype, seed=18, gamma=(0.97, 0.999))
    got, fin = run_gpu(x, chunk=128, return_final_state=True)
    # widths round the sums differently, so only the width the call ran at matches bit for bit
    same = []
    for W in (64, 32, 16):
        o, f = run_gpu(x, chunk=W, return_final_state=True)
        if torch.equal(o, got):
            same.append((W, f))
    assert same, "the call at chunk 128 matches no narrower width"
    W, f = same[0]
    got_f, want_f = O.unpack_state(np64(fin.cpu()), d, dv), O.unpack_state(np64(f.cpu()), d, dv)
    for key in ("S", "C", "m", "G", "h"):
        assert rel_err(got_f[key], want_f[key]) <= 1e-4, key
    # the queries for the same call (with a final state) as the one compared above
    assert hla.forward_plan(1, 3, 1000, d, dv, 128, dtype, want_final_state=True) == \
        hla.forward_plan(1, 3, 1000, d, dv, W, dtype, want_final_state=True)
    assert hla.forward_workspace_bytes(1, 3, 1000, d, dv, 128, dtype, want_final_state=True) == \
        hla.forward_workspace_bytes(1, 3, 1000, d, dv, W, dtype, want_final_state=True)
    ref, ref_state = oracle(x, return_state=True)
    assert rel_err(np64(got.cpu()), ref) <= tol_for(dtype)
    got_s, want_s = O.unpack_state(np64(fin.cpu()), d, dv), O.unpack_state(ref_state, d, dv)
    for key in ("S", "C", "m", "G", "h"):
        assert rel_err(got_s[key], want_s[key]) <= tol_for(dtype), key


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_normalized_with_decay(dtype):
    x = inputs.make_custom(2, 2, 300, 32, 32, dtype, seed=14, qk="softplus", v_scale="unit",
                           gamma=(0.95, 0.999))
    o = run_gpu(x, chunk=32, normalize=True, eps=1e-6).cpu()
    assert rel_err(np64(o), oracle(x, normalize=True)) <= tol_for(dtype)


# ---- state in and out -----------------------------------------------------------------------

@pytest.mark.parametrize("dtype, d", [(torch.float32, 16), (torch.bfloat16, 64), (torch.bfloat16, 128)])
def test_final_state_matches_oracle(dtype, d):
    x = inputs.make_custom(1, 2, 5 * 64 + 9, d, d, dtype, seed=15, gamma=(0.97, 0.999))
    o, fin = run_gpu(x, chunk=64 if d > 16 else 16, return_final_state=True)
    ref, ref_state = oracle(x, return_state=True)
    assert rel_err(np64(o.cpu()), ref) <= tol_for(dtype)
    got = O.unpack_state(np64(fin.cpu()), d, d)
    want = O.unpack_state(ref_state, d, d)
    for key in ("S", "C", "m", "G", "h"):
        assert rel_err(got[key], want[key]) <= tol_for(dtype), key


@pytest.mark.parametrize("dtype, d", [(torch.float32, 32), (torch.bfloat16, 64)])
def test_continuation_from_init_state(dtype, d):
    """Forward over [0, n) equals forward over [0, m) then [m, n) from its final state."""
    x = inputs.make_custom(2, 2, 700, d, d, dtype, seed=16, gamma=(0.99, 0.999))
    m = 300
    first = {key: (val[:, :, :m].contiguous() if key in ("q", "k", "v") else val) for key, val in x.items()}
    second = {key: (val[:, :, m:].contiguous() if key in ("q", "k", "v") else val) for key, val in x.items()}
    _, s1 = run_gpu(first, chunk=32, return_final_state=True)
    o2 = run_gpu(second, chunk=32, init_state=s1).cpu()
    ref = oracle(x)[:, :, m:]
    assert rel_err(np64(o2), ref) <= tol_for(dtype)


def test_empty_sequence_passes_state_through():
    x = inputs.make_custom(1, 2, 0, 16, 16, torch.float32, seed=17, gamma=0.9)
    init = torch.randn(1, 2, hla.state_floats(16, 16))
    o, fin = run_gpu(x, chunk=16, init_state=init.cuda(), return_final_state=True)
    assert o.shape == (1, 2, 0, 16)
    assert torch.equal(fin.cpu(), init)


def test_causality_on_gpu():
    x = inputs.make_custom(1, 2, 500, 64, 64, torch.bfloat16, seed=18, gamma=0.99)
    o1 = run_gpu(x, chunk=64).cpu()
    y = dict(x)
    y["q"] = x["q"].clone()
    y["k"] = x["k"].clone()
    y["v"] = x["v"].clone()
    y["q"][:, :, 300:] = torch.randn_like(y["q"][:, :, 300:].float()).to(torch.bfloat16)
    y["v"][:, :, 300:] = 0
    o2 = run_gpu(y, chunk=64).cpu()
    assert torch.equal(o1[:, :, :300], o2[:, :, :300])


def test_host_tensors_round_trip():
    """CPU tensors in, CPU tensor out (the end-to-end path of the binding)."""
    x = inputs.make_custom(1, 2, 130, 32, 32, torch.bfloat16, seed=19, gamma=0.98)
    o = hla.forward(x["q"].pin_memory(), x["k"].pin_memory(), x["v"].pin_memory(), gamma=x["gamma"],
                    chunk=32)
    assert o.device.type == "cpu"
    assert rel_err(np64(o), oracle(x)) <= 2e-2


@pytest.mark.parametrize("B,H,chunk", [(2, 8, 64), (1, 16, 128), (3, 4, 32)])
def test_host_tensors_pipelined_by_head_groups(B, H, chunk):
    """Host tensors go through in head groups (copies overlapped with the computation):
    the result matches the oracle and the all-device call, with and without an out buffer."""
    x = inputs.make_custom(B, H, 700, 64, 64, torch.bfloat16, seed=23 + H, gamma=(0.95, 0.999))
    ref = oracle(x)
    o = hla.forward(x["q"].pin_memory(), x["k"].pin_memory(), x["v"].pin_memory(), gamma=x["gamma"].cuda(),
                    chunk=chunk)
    assert o.device.type == "cpu" and rel_err(np64(o), ref) <= 2e-2
    buf = torch.empty_like(x["v"]).pin_memory()
    o2 = hla.forward(x["q"].pin_memory(), x["k"].pin_memory(), x["v"].pin_memory(), gamma=x["gamma"].cuda(),
                     chunk=chunk, out=buf)
    assert o2.data_ptr() == buf.data_ptr() and torch.equal(o2, o)
    dev = run_gpu(x, chunk=chunk).cpu()
    assert rel_err(np64(o), np64(dev)) <= 2e-2


def test_workspace_too_small_is_reported():
    import ctypes
    x = inputs.make_custom(1, 1, 64, 16, 16, torch.bfloat16, seed=20)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    out = torch.empty_like(v)
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    opts = hla.hla2.Opts(1, 1e-6, ws.data_ptr(), 16, None, None)
    rc = hla.lib().hla2_forward(*(ctypes.c_void_p(t.data_ptr()) for t in (q, k, v, out)), 1, 1, 64, 16, 16,
                                None, 0, 16, None, ctypes.byref(opts))
    assert rc == -3
