"""The bf16 training path (d = dv = 128 and 64) on the tcgen05 first-order scan kernels (chunk
128), and the d = 128 forward (plain, or with the final state) on the same passes, through the
C ABI, against the float64 oracle.

The masked output is two chained first-order scans (p = S q, then o = q^T Z) and its reverse
mode six more; every pass runs segment-parallel on the same kernel.  Bar: max|gpu - oracle| /
max|oracle| <= 2e-2 per gradient and for the output (bf16 inputs; the oracle runs on the same
bf16-rounded values).  Sizes span one and many segments, multi-chunk segments, ragged tails
(the last chunk partial), a sequence shorter than a chunk, one token, and no decay.
"""
import os

import numpy as np
import pytest
import torch

import chunked_scan_mixer_gb300 as hla
from chunked_scan_mixer_gb300 import inputs
from oracle import ahla_oracle as A
from oracle import cref

from .helpers import np32, np64, rel_err

pytestmark = pytest.mark.gpu

D = 128


def _gamma_np(x):
    return None if x["gamma"] is None else x["gamma"].double().numpy()


def _dev(x):
    g = None if x["gamma"] is None else x["gamma"].cuda()
    return x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["dout"].cuda(), g


def _check_grads(got, x, what=""):
    ref = cref.backward(np32(x["q"]), np32(x["k"]), np32(x["v"]), np32(x["dout"]), _gamma_np(x))
    for name, gg, rr in zip(("dq", "dk", "dv"), got, ref):
        assert torch.isfinite(gg.float()).all(), (name, what)
        err = rel_err(np64(gg.cpu()), rr)
        assert err <= 2e-2, (name, what, err)


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("B, H, n", [(1, 2, 1000), (2, 8, 4000), (1, 3, 128), (1, 2, 127), (1, 2, 129),
                                     (1, 1, 1), (3, 1, 2500)])
@pytest.mark.parametrize("gamma", [None, (0.9, 0.999)])
def test_backward_matches_oracle(d, B, H, n, gamma):
    x = inputs.make_custom(B, H, n, d, d, torch.bfloat16, seed=B * 1000 + H * 100 + n % 97 + d, gamma=gamma,
                           with_dout=True)
    q, k, v, do, g = _dev(x)
    _check_grads(hla.backward(q, k, v, do, gamma=g, chunk=128), x, (B, H, n, gamma))


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("n", [300, 3000])
def test_forward_saved_then_backward(d, n):
    """The forward that keeps p for the backward gives the oracle's output; the backward from
    the saved p and carries equals, bit for bit, the one that recomputes them, and the oracle."""
    x = inputs.make_custom(2, 3, n, d, d, torch.bfloat16, seed=n + d, gamma=(0.97, 0.999), with_dout=True)
    q, k, v, do, g = _dev(x)
    o, saved = hla.forward(q, k, v, gamma=g, chunk=128, save_for_backward=True)
    ref = cref.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), _gamma_np(x))
    assert rel_err(np64(o.cpu()), ref) <= 2e-2
    plain = hla.forward(q, k, v, gamma=g, chunk=128)
    assert rel_err(np64(o.cpu()), np64(plain.cpu())) <= 2e-2
    a = hla.backward(q, k, v, do, gamma=g, chunk=128, saved=saved)
    b = hla.backward(q, k, v, do, gamma=g, chunk=128)
    for u, w in zip(a, b):
        assert torch.equal(u, w)
    _check_grads(a, x, "saved")


@pytest.mark.parametrize("d", [128, 64])
def test_steep_and_flat_decay_per_head(d):
    """Decays from 0.5 (a pair weight that underflows within a chunk) to 1 across heads."""
    x = inputs.make_custom(1, 4, 700, d, d, torch.bfloat16, seed=77, gamma=None, with_dout=True)
    x["gamma"] = torch.tensor([0.5, 0.9, 0.999, 1.0], dtype=torch.float32)
    q, k, v, do, g = _dev(x)
    _check_grads(hla.backward(q, k, v, do, gamma=g, chunk=128), x)


def test_training_workload_all_heads():
    """B=4, H=16, n=8192, d=dv=128, decay 0.995: forward keeping p, then the backward from it;
    the output and all 64 heads' gradients against the oracle."""
    w = inputs.WORKLOADS["train"]
    assert w.chunk == 128
    x = inputs.make(w)
    q, k, v, do, g = _dev(x)
    o, saved = hla.forward(q, k, v, gamma=g, chunk=w.chunk, save_for_backward=True)
    grads = hla.backward(q, k, v, do, gamma=g, chunk=w.chunk, saved=saved)
    torch.cuda.synchronize()
    ref_o = cref.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), _gamma_np(x))
    assert rel_err(np64(o.cpu()), ref_o) <= 2e-2
    del ref_o
    ref = cref.backward(np32(x["q"]), np32(x["k"]), np32(x["v"]), np32(x["dout"]), _gamma_np(x))
    for name, gg, rr in zip(("dq", "dk", "dv"), grads, ref):
        got = np64(gg.cpu())
        assert rel_err(got, rr) <= 2e-2, name
        per_head = [rel_err(got[b, h], rr[b, h]) for b in range(w.B) for h in range(w.H)]
        assert max(per_head) <= 2e-2, (name, int(np.argmax(per_head)))


@pytest.mark.parametrize("d", [128, 64])
def test_distinct_from_the_legacy_path(d):
    """HLA2_KERNEL=mma selects the mma.sync kernels: both paths match the oracle, and their
    gradients are not bit for bit equal (different kernels, different rounding order), so the
    default call does run the first-order scan kernels."""
    x = inputs.make_custom(1, 2, 600, d, d, torch.bfloat16, seed=5 + d, gamma=(0.98, 0.999), with_dout=True)
    q, k, v, do, g = _dev(x)
    tc = hla.backward(q, k, v, do, gamma=g, chunk=128)
    old = os.environ.get("HLA2_KERNEL")
    os.environ["HLA2_KERNEL"] = "mma"
    try:
        legacy = hla.backward(q, k, v, do, gamma=g, chunk=128)
    finally:
        if old is None:
            os.environ.pop("HLA2_KERNEL", None)
        else:
            os.environ["HLA2_KERNEL"] = old
    _check_grads(tc, x, "tcgen05")
    _check_grads(legacy, x, "mma.sync")
    assert not all(torch.equal(a, b) for a, b in zip(tc, legacy))


# (2, 25, 2100): 3 segments of 6 chunks per head, the last chunk ragged, so that every
# pipeline's stages are reused within a segment and carries cross the segments
@pytest.mark.parametrize("B, H, n", [(1, 2, 1000), (2, 3, 129), (1, 1, 1), (1, 4, 3000), (2, 25, 2100)])
@pytest.mark.parametrize("gamma", [None, (0.9, 0.999)])
def test_forward_matches_oracle(B, H, n, gamma):
    """The plain forward (no state in or out) runs the same first-order passes."""
    x = inputs.make_custom(B, H, n, D, D, torch.bfloat16, seed=7 * n + H, gamma=gamma)
    g = None if x["gamma"] is None else x["gamma"].cuda()
    o = hla.forward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), gamma=g, chunk=128)
    ref = cref.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), _gamma_np(x))
    assert rel_err(np64(o.cpu()), ref) <= 2e-2
    nseg, seg_chunks, launches = hla.forward_plan(B, H, n, D, D, 128)
    assert launches == 6 + (2 if nseg > 1 else 0) and nseg * seg_chunks * 128 >= n


def test_forward_distinct_from_the_legacy_path():
    x = inputs.make_custom(1, 2, 700, D, D, torch.bfloat16, seed=9, gamma=(0.98, 0.999))
    q, k, v, g = x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["gamma"].cuda()
    tc = hla.forward(q, k, v, gamma=g, chunk=128)
    old = os.environ.get("HLA2_KERNEL")
    os.environ["HLA2_KERNEL"] = "mma"
    try:
        legacy = hla.forward(q, k, v, gamma=g, chunk=128)
    finally:
        if old is None:
            os.environ.pop("HLA2_KERNEL", None)
        else:
            os.environ["HLA2_KERNEL"] = old
    ref = cref.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), _gamma_np(x))
    assert rel_err(np64(tc.cpu()), ref) <= 2e-2 and rel_err(np64(legacy.cpu()), ref) <= 2e-2
    assert not torch.equal(tc, legacy)


@pytest.mark.parametrize("B, H, n", [(1, 2, 1000), (2, 3, 129), (1, 1, 1), (1, 4, 3000), (2, 64, 700),
                                     (2, 25, 2100)])
@pytest.mark.parametrize("gamma", [None, (0.9, 0.999)])
def test_forward_final_state_matches_oracle(B, H, n, gamma):
    """The d = 128 forward with the state after the last token, on the first-order scans: the
    (q, v) summaries, the m and y moments (y from the stored full p), the carries into the last
    segment, and its combine.  Every part (S, C, m, G, h) and the output against the oracle, on
    one and many segments per head (B H = 128: one each), ragged tails, one token."""
    x = inputs.make_custom(B, H, n, D, D, torch.bfloat16, seed=11 * n + H, gamma=gamma)
    g = None if x["gamma"] is None else x["gamma"].cuda()
    o, fin = hla.forward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), gamma=g, chunk=128, return_final_state=True)
    hla.check_status()
    ref, ref_state = cref.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), _gamma_np(x), return_state=True)
    assert rel_err(np64(o.cpu()), ref) <= 2e-2
    from oracle import hla2_oracle as O
    got, want = O.unpack_state(np64(fin.cpu()), D, D), O.unpack_state(ref_state, D, D)
    for key in ("S", "C", "m", "G", "h"):
        assert rel_err(got[key], want[key]) <= 2e-2, key
    nseg, seg_chunks, launches = hla.forward_plan(B, H, n, D, D, 128, want_final_state=True)
    assert launches == 7 + (3 if nseg > 1 else 0)


def test_final_state_then_decode_and_distinct_from_the_legacy_path():
    """A d = 128 prefill on the first-order scans, then decode steps from its state, against the
    oracle over the whole sequence; the same prefill on the mma.sync kernels meets the bar with
    other bits."""
    B, H, n, steps = 2, 4, 128 * 12 + 37, 3
    x = inputs.make_custom(B, H, n + steps, D, D, torch.bfloat16, seed=61, gamma=(0.99, 0.9995))
    g = x["gamma"].cuda()
    part = lambda lo, hi: [x[t][:, :, lo:hi].contiguous().cuda() for t in ("q", "k", "v")]
    o, fin = hla.forward(*part(0, n), gamma=g, chunk=128, return_final_state=True)
    old = os.environ.get("HLA2_KERNEL")
    os.environ["HLA2_KERNEL"] = "mma"
    try:
        o2, fin2 = hla.forward(*part(0, n), gamma=g, chunk=128, return_final_state=True)
    finally:
        if old is None:
            os.environ.pop("HLA2_KERNEL", None)
        else:
            os.environ["HLA2_KERNEL"] = old
    assert not torch.equal(fin, fin2)
    ref = cref.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), _gamma_np(x))
    assert rel_err(np64(o.cpu()), ref[:, :, :n]) <= 2e-2 and rel_err(np64(o2.cpu()), ref[:, :, :n]) <= 2e-2
    for t in range(n, n + steps):
        q, k, v = part(t, t + 1)
        y = hla.decode_step(fin, q[:, :, 0], k[:, :, 0], v[:, :, 0], gamma=g)
        assert rel_err(np64(y.cpu()), ref[:, :, t]) <= 2e-2, t


def test_d64_training_shapes_all_heads():
    """The training workload's batch and length at d = dv = 64 (B=4, H=16, n=8192): forward
    keeping p, backward from it; output and all 64 heads' gradients against the oracle."""
    w = inputs.WORKLOADS["train"]
    x = inputs.make_custom(w.B, w.H, w.n, 64, 64, torch.bfloat16, seed=55, gamma=0.995, with_dout=True)
    q, k, v, do, g = _dev(x)
    o, saved = hla.forward(q, k, v, gamma=g, chunk=128, save_for_backward=True)
    grads = hla.backward(q, k, v, do, gamma=g, chunk=128, saved=saved)
    torch.cuda.synchronize()
    assert rel_err(np64(o.cpu()), cref.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), _gamma_np(x))) <= 2e-2
    ref = cref.backward(np32(x["q"]), np32(x["k"]), np32(x["v"]), np32(x["dout"]), _gamma_np(x))
    for name, gg, rr in zip(("dq", "dk", "dv"), grads, ref):
        got = np64(gg.cpu())
        per_head = [rel_err(got[b, h], rr[b, h]) for b in range(w.B) for h in range(w.H)]
        assert max(per_head) <= 2e-2, (name, int(np.argmax(per_head)))


# ---- AHLA reverse mode (d = dv = 64, chunk 128) on the same kernel -----------------------------

def _ahla_grads(x, chunk=128):
    g = None if x["gamma"] is None else x["gamma"].cuda()
    return hla.ahla_backward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["dout"].cuda(), gamma=g, chunk=chunk)


@pytest.mark.parametrize("B, H, n", [(1, 2, 1000), (2, 3, 129), (1, 1, 1), (1, 2, 127), (2, 8, 3000)])
@pytest.mark.parametrize("gamma", [None, (0.9, 0.999)])
def test_ahla_backward_matches_oracle(B, H, n, gamma):
    """AHLA gradients (u = LA(q, k, v), o = LA(q, k, u) and six reverse-mode scans) against the
    oracle's reverse sweep of the AHLA streaming recurrence."""
    x = inputs.make_custom(B, H, n, 64, 64, torch.bfloat16, seed=11 * n + H, gamma=gamma, with_dout=True)
    got = _ahla_grads(x)
    ref = A.serial_backward(np32(x["q"]), np32(x["k"]), np32(x["v"]), np32(x["dout"]), _gamma_np(x))
    for name, gg, rr in zip(("dq", "dk", "dv"), got, ref):
        assert torch.isfinite(gg.float()).all(), name
        assert rel_err(np64(gg.cpu()), rr) <= 2e-2, (name, B, H, n, gamma)


def test_ahla_backward_long_context_sampled_heads():
    """The AHLA backward at the long-context shapes (B=1 H=16 n=65536 d=dv=64 bf16, decay
    linspace(0.99, 0.9999), chunk 128), the launch configuration of the bench's row (dk and dq
    each one pass over two stacked query / key pairs): heads 0 and 15, the fastest and the
    slowest decay (whose carries reach furthest across segments), against the oracle's reverse
    sweep of the whole sequence."""
    import dataclasses

    w = dataclasses.replace(inputs.WORKLOADS["long"], with_dout=True)
    x = inputs.make(w, seed=w.seed + 7)
    got = [t.cpu() for t in _ahla_grads(x)]
    g = _gamma_np(x)
    for h in (0, w.H - 1):
        sl = slice(h, h + 1)
        ref = A.serial_backward(np32(x["q"][:, sl]), np32(x["k"][:, sl]), np32(x["v"][:, sl]),
                                np32(x["dout"][:, sl]), g[sl])
        for name, gg, rr in zip(("dq", "dk", "dv"), got, ref):
            assert rel_err(np64(gg[:, sl]), rr) <= 2e-2, (name, h)


def test_ahla_backward_distinct_from_the_simt_path():
    x = inputs.make_custom(1, 2, 600, 64, 64, torch.bfloat16, seed=12, gamma=(0.97, 0.999), with_dout=True)
    tc = _ahla_grads(x)
    old = os.environ.get("HLA2_KERNEL")
    os.environ["HLA2_KERNEL"] = "mma"
    try:
        simt = _ahla_grads(x)
    finally:
        if old is None:
            os.environ.pop("HLA2_KERNEL", None)
        else:
            os.environ["HLA2_KERNEL"] = old
    ref = A.serial_backward(np32(x["q"]), np32(x["k"]), np32(x["v"]), np32(x["dout"]), _gamma_np(x))
    for gg in (tc, simt):
        for name, g1, rr in zip(("dq", "dk", "dv"), gg, ref):
            assert rel_err(np64(g1.cpu()), rr) <= 2e-2, name
    assert not all(torch.equal(a, b) for a, b in zip(tc, simt))
