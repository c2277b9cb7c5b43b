"""The tcgen05 chunk kernels (bf16, d = dv = 64, chunk 128) against the float64
oracle and against the mma.sync chunk kernels on the same inputs, through the C ABI."""
import os

import pytest
import torch

import chunked_scan_mixer_gb300 as hla
from chunked_scan_mixer_gb300 import inputs
from oracle import cref

from .helpers import np32, np64, rel_err

pytestmark = pytest.mark.gpu


def run(x, kernel=None, **kw):
    old = os.environ.pop("HLA2_KERNEL", None)
    if kernel:
        os.environ["HLA2_KERNEL"] = kernel
    try:
        g = None if x["gamma"] is None else x["gamma"].cuda()
        o = hla.forward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), gamma=g, chunk=128, **kw)
        hla.check_status()
        return o.cpu() if torch.is_tensor(o) else tuple(t.cpu() for t in o)
    finally:
        os.environ.pop("HLA2_KERNEL", None)
        if old is not None:
            os.environ["HLA2_KERNEL"] = old


def oracle(x, **kw):
    g = None if x["gamma"] is None else x["gamma"].double().numpy()
    return cref.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), g, **kw)


@pytest.mark.parametrize("n", [1, 64, 127, 128, 129, 300, 1000, 4096 + 33])
def test_lengths(n):
    x = inputs.make_custom(1, 3, n, 64, 64, torch.bfloat16, seed=n, gamma=(0.97, 0.9999))
    o = run(x)
    assert torch.isfinite(o.float()).all()
    assert rel_err(np64(o), oracle(x)) <= 2e-2


@pytest.mark.parametrize("gamma", [None, 0.9, (0.5, 0.999)])
def test_decays(gamma):
    x = inputs.make_custom(2, 2, 700, 64, 64, torch.bfloat16, seed=7, gamma=gamma)
    assert rel_err(np64(run(x)), oracle(x)) <= 2e-2


def test_matches_mma_path():
    x = inputs.make_custom(1, 4, 2000, 64, 64, torch.bfloat16, seed=8, gamma=(0.99, 0.9999))
    a = np64(run(x))
    b = np64(run(x, kernel="mma"))
    ref = oracle(x)
    assert rel_err(a, ref) <= 2e-2 and rel_err(b, ref) <= 2e-2
    assert rel_err(a, b) <= 2e-2


def test_many_heads_one_segment_each():
    x = inputs.make_custom(4, 80, 256, 64, 64, torch.bfloat16, seed=9, gamma=0.995)
    o = run(x)
    ref = oracle(x)
    assert rel_err(np64(o), ref) <= 2e-2


def test_repeated_calls_are_identical():
    x = inputs.make_custom(1, 2, 1500, 64, 64, torch.bfloat16, seed=10, gamma=(0.98, 0.999))
    a, b = run(x), run(x)
    assert torch.equal(a, b)


@pytest.mark.parametrize("B,H,n", [(4, 80, 128 * 40), (1, 16, 128 * 60 + 77), (1, 8, 128 * 100 + 1), (1, 2, 128 * 500 + 64)])
def test_multi_chunk_segments(B, H, n):
    """Segments of several chunks (odd and even counts, ragged last chunk): exercises the
    double-buffered key loads and the carried state inside one CTA."""
    nseg, seg_chunks, _ = hla.forward_plan(B, H, n, 64, 64, 128)
    assert seg_chunks >= 3
    x = inputs.make_custom(B, H, n, 64, 64, torch.bfloat16, seed=n % 1000, gamma=(0.98, 0.9999))
    assert rel_err(np64(run(x)), oracle(x)) <= 2e-2


@pytest.mark.parametrize("gamma", [None, (0.5, 0.9)])
def test_multi_chunk_segments_decay_extremes(gamma):
    """Segments of several chunks without decay and with strong decay: on the stored-p path
    the carry enters each chunk as g^(it W + r + 1) S_in q, which underflows to zero within a
    chunk or two at g = 0.5 (exactly the weight the pair sum gives it)."""
    B, H, n = 1, 16, 128 * 40 + 9
    nseg, seg_chunks, _ = hla.forward_plan(B, H, n, 64, 64, 128)
    assert nseg > 1 and seg_chunks >= 2
    x = inputs.make_custom(B, H, n, 64, 64, torch.bfloat16, seed=31, gamma=gamma)
    o = run(x)
    assert torch.isfinite(o.float()).all()
    assert rel_err(np64(o), oracle(x)) <= 2e-2


def _device_inputs(seed, B=1, H=16, n=128 * 40 + 9):
    x = inputs.make_custom(B, H, n, 64, 64, torch.bfloat16, seed=seed, gamma=(0.98, 0.9999))
    return x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["gamma"].cuda()


def test_graph_capture_replays_forward():
    """The stored-p forward (kernels chained by programmatic dependent launch) captured in a CUDA
    graph: a replay reproduces the eager output bit for bit, and a replay after new inputs are
    written into the captured buffers recomputes."""
    q, k, v, g = _device_inputs(33)
    ref = hla.forward(q, k, v, gamma=g, chunk=128)
    out = torch.empty_like(v)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture
        hla.forward(q, k, v, gamma=g, chunk=128, out=out)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        hla.forward(q, k, v, gamma=g, chunk=128, out=out)
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    q2, k2, v2, _ = _device_inputs(34)
    ref2 = hla.forward(q2, k2, v2, gamma=g, chunk=128)
    q.copy_(q2)
    k.copy_(k2)
    v.copy_(v2)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref2)


def test_concurrent_streams():
    """Two forwards in flight on two streams at once (each stream has its own workspace)."""
    xs = [_device_inputs(35), _device_inputs(36)]
    refs = [hla.forward(q, k, v, gamma=g, chunk=128) for q, k, v, g in xs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for (q, k, v, g), s in zip(xs, streams):
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            outs.append(hla.forward(q, k, v, gamma=g, chunk=128))
    torch.cuda.synchronize()
    for o, r in zip(outs, refs):
        assert torch.equal(o, r)


@pytest.mark.parametrize("masked", [True, False])
def test_stored_p_path_continues_from_init_state(masked):
    """The stored-p kernels with a carried-in state: a prefill over [0, m) (final state on the
    mma.sync path), then [m, n) at chunk 128 on multi-chunk segments from that state, equals the
    oracle over [0, n) on the second part.  Segment 0's carry is then nonzero, so its
    Q S_in term and Z_in enter as well."""
    B, H, m, n2 = 1, 16, 300, 128 * 40 + 9
    nseg, seg_chunks, _ = hla.forward_plan(B, H, n2, 64, 64, 128)
    assert nseg > 1 and seg_chunks >= 2
    x = inputs.make_custom(B, H, m + n2, 64, 64, torch.bfloat16, seed=37, gamma=(0.98, 0.9999))
    g = x["gamma"].cuda()
    part = lambda lo, hi: [x[t][:, :, lo:hi].contiguous().cuda() for t in ("q", "k", "v")]
    _, s1 = hla.forward(*part(0, m), gamma=g, chunk=32, return_final_state=True, masked=masked)
    o2 = hla.forward(*part(m, m + n2), gamma=g, chunk=128, init_state=s1, masked=masked)
    hla.check_status()
    gd = x["gamma"].double().numpy()
    ref = cref.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), gd, masked=masked)[:, :, m:]
    assert rel_err(np64(o2.cpu()), ref) <= 2e-2


def _unpack(state, d=64):
    from oracle import hla2_oracle as O
    return O.unpack_state(np64(state.cpu()), d, d)


@pytest.mark.parametrize("B,H,n", [(1, 16, 128 * 40 + 9), (1, 8, 128 * 100 + 1), (2, 8, 100)])
def test_final_state_on_the_stored_p_path(B, H, n):
    """The state after the last token from the tcgen05 path (summaries of every segment, their
    q and p moments, the carry into the last segment combined with its summary): every part
    (S, C, m, G, h) and the output against the oracle, on multi-segment and one-segment calls."""
    x = inputs.make_custom(B, H, n, 64, 64, torch.bfloat16, seed=41 + H, gamma=(0.97, 0.9999))
    g = x["gamma"].cuda()
    o, fin = hla.forward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), gamma=g, chunk=128, return_final_state=True)
    hla.check_status()
    gd = x["gamma"].double().numpy()
    ref, ref_state = cref.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), gd, return_state=True)
    assert rel_err(np64(o.cpu()), ref) <= 2e-2
    from oracle import hla2_oracle as O
    got, want = _unpack(fin), O.unpack_state(ref_state, 64, 64)
    for key in ("S", "C", "m", "G", "h"):
        assert rel_err(got[key], want[key]) <= 2e-2, key


def test_final_state_with_init_state_and_decode_after():
    """Prefill at chunk 128 from a carried-in state, with the final state; the decode steps that
    follow match the oracle run over the whole sequence."""
    B, H, m, n2, steps = 1, 16, 300, 128 * 40 + 9, 3
    x = inputs.make_custom(B, H, m + n2 + steps, 64, 64, torch.bfloat16, seed=43, gamma=(0.98, 0.9999))
    g = x["gamma"].cuda()
    part = lambda lo, hi: [x[t][:, :, lo:hi].contiguous().cuda() for t in ("q", "k", "v")]
    _, s1 = hla.forward(*part(0, m), gamma=g, chunk=32, return_final_state=True)
    o2, s2 = hla.forward(*part(m, m + n2), gamma=g, chunk=128, init_state=s1, return_final_state=True)
    hla.check_status()
    gd = x["gamma"].double().numpy()
    ref = cref.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), gd)
    assert rel_err(np64(o2.cpu()), ref[:, :, m:m + n2]) <= 2e-2
    for t in range(m + n2, m + n2 + steps):
        q, k, v = part(t, t + 1)
        o = hla.decode_step(s2, q[:, :, 0], k[:, :, 0], v[:, :, 0], gamma=g)
        assert rel_err(np64(o.cpu()), ref[:, :, t]) <= 2e-2, t


def test_final_state_paths_agree():
    """tcgen05 and mma.sync final states on the same inputs."""
    x = inputs.make_custom(2, 8, 128 * 24 + 5, 64, 64, torch.bfloat16, seed=45, gamma=(0.99, 0.9999))
    g = x["gamma"].cuda()
    args = (x["q"].cuda(), x["k"].cuda(), x["v"].cuda())
    _, a = hla.forward(*args, gamma=g, chunk=128, return_final_state=True)
    old = os.environ.pop("HLA2_KERNEL", None)
    os.environ["HLA2_KERNEL"] = "mma"
    try:
        _, b = hla.forward(*args, gamma=g, chunk=128, return_final_state=True)
    finally:
        os.environ.pop("HLA2_KERNEL", None)
        if old is not None:
            os.environ["HLA2_KERNEL"] = old
    ga, gb = _unpack(a), _unpack(b)
    for key in ("S", "C", "m", "G", "h"):
        assert rel_err(ga[key], gb[key]) <= 2e-2, key


# ---- ratio-normalised output on the stored-p kernels ---------------------------------------

def test_normalized_workload_at_chunk_128():
    """The normalised workload (B=2 H=8 n=2048, softplus features, decay linspace(0.95, 0.999))
    at chunk 128: the tcgen05 stored-p kernels, whose output pass forms the denominator rows
    and the y moment in its epilogue.  Against the oracle, reproducible bit for bit, and other
    bits than the mma.sync kernels give on the same inputs (which also meet the bar)."""
    x = inputs.make("normed")
    a = run(x, normalize=True, eps=x["eps"])
    ref = oracle(x, normalize=True, eps=x["eps"])
    assert torch.isfinite(a.float()).all()
    assert rel_err(np64(a), ref) <= 2e-2
    assert torch.equal(a, run(x, normalize=True, eps=x["eps"]))
    b = run(x, kernel="mma", normalize=True, eps=x["eps"])
    assert rel_err(np64(b), ref) <= 2e-2
    assert not torch.equal(a, b)


@pytest.mark.parametrize("B,H,n", [(1, 16, 128 * 40 + 9), (1, 2, 100), (2, 3, 1000), (1, 4, 128)])
def test_normalized_lengths_and_segments(B, H, n):
    """One-segment calls (the summary pass then only stores p) and multi-segment calls (the y
    carry from the segment moments, cross terms and scan), ragged tails, a single chunk."""
    x = inputs.make_custom(B, H, n, 64, 64, torch.bfloat16, seed=50 + n % 97, qk="softplus", v_scale="unit",
                           gamma=(0.95, 0.999))
    o = run(x, normalize=True)
    assert rel_err(np64(o), oracle(x, normalize=True)) <= 2e-2


@pytest.mark.parametrize("gamma", [None, 0.9, (0.5, 0.9999)])
def test_normalized_decays(gamma):
    x = inputs.make_custom(2, 4, 1500, 64, 64, torch.bfloat16, seed=53, qk="softplus", v_scale="unit", gamma=gamma)
    assert rel_err(np64(run(x, normalize=True)), oracle(x, normalize=True)) <= 2e-2


def test_normalized_with_init_state_and_final_state():
    """A normalised prefill continued from a carried-in state (segment 0's y carry nonzero),
    returning the final state: the output over the second part and every part of the state
    against the oracle over the whole sequence."""
    B, H, m, n2 = 1, 16, 300, 128 * 30 + 17
    x = inputs.make_custom(B, H, m + n2, 64, 64, torch.bfloat16, seed=57, qk="softplus", v_scale="unit",
                           gamma=(0.97, 0.9999))
    g = x["gamma"].cuda()
    part = lambda lo, hi: [x[t][:, :, lo:hi].contiguous().cuda() for t in ("q", "k", "v")]
    _, s1 = hla.forward(*part(0, m), gamma=g, chunk=32, normalize=True, return_final_state=True)
    o2, s2 = hla.forward(*part(m, m + n2), gamma=g, chunk=128, normalize=True, init_state=s1,
                         return_final_state=True)
    hla.check_status()
    gd = x["gamma"].double().numpy()
    ref, ref_state = cref.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), gd, normalize=True, return_state=True)
    assert rel_err(np64(o2.cpu()), ref[:, :, m:]) <= 2e-2
    from oracle import hla2_oracle as O
    got, want = _unpack(s2), O.unpack_state(ref_state, 64, 64)
    for key in ("S", "C", "m", "G", "h"):
        assert rel_err(got[key], want[key]) <= 2e-2, key
