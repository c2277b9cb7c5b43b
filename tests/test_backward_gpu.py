"""GPU reverse-mode chunk scan (dQ, dK, dV) against the float64 oracle's reverse sweep of
the serial recurrence, through the C ABI.  Bar: max|gpu - oracle| / max|oracle| <= 2e-2
per gradient for bf16 inputs (the oracle runs on the same bf16-rounded values) and <= 1e-4
for float32 inputs (the SIMT float32 kernels, any d and dv)."""
import numpy as np
import pytest
import torch

import chunked_scan_mixer_gb300 as hla
from chunked_scan_mixer_gb300 import HLA2Error, inputs
from oracle import cref

from .helpers import np32, np64, rel_err

pytestmark = pytest.mark.gpu


def run(x, chunk):
    g = None if x["gamma"] is None else x["gamma"].cuda()
    return hla.backward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["dout"].cuda(), gamma=g, chunk=chunk)


def oracle(x):
    g = None if x["gamma"] is None else x["gamma"].double().numpy()
    return cref.backward(np32(x["q"]), np32(x["k"]), np32(x["v"]), np32(x["dout"]), g)


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("chunk", [16, 32, 64])
def test_gradients_match_oracle(d, chunk):
    n = 3 * chunk + 7
    x = inputs.make_custom(1, 3, n, d, d, torch.bfloat16, seed=d * 7 + chunk, gamma=(0.9, 0.999),
                           with_dout=True)
    got = run(x, chunk)
    ref = oracle(x)
    for name, gg, rr in zip(("dq", "dk", "dv"), got, ref):
        assert torch.isfinite(gg.float()).all(), name
        assert rel_err(np64(gg.cpu()), rr) <= 2e-2, name


@pytest.mark.parametrize("n", [1, 5, 64, 200, 1000])
def test_lengths_and_segments(n):
    x = inputs.make_custom(2, 2, n, 64, 64, torch.bfloat16, seed=n, gamma=(0.95, 0.995), with_dout=True)
    got = run(x, 64)
    ref = oracle(x)
    for name, gg, rr in zip(("dq", "dk", "dv"), got, ref):
        assert rel_err(np64(gg.cpu()), rr) <= 2e-2, (name, n)


def test_no_decay():
    x = inputs.make_custom(1, 2, 500, 32, 32, torch.bfloat16, seed=3, gamma=None, with_dout=True)
    got = run(x, 32)
    ref = oracle(x)
    for gg, rr in zip(got, ref):
        assert rel_err(np64(gg.cpu()), rr) <= 2e-2


def test_chunk_width_independence():
    x = inputs.make_custom(1, 2, 333, 64, 64, torch.bfloat16, seed=4, gamma=(0.97, 0.999), with_dout=True)
    a = [np64(t.cpu()) for t in run(x, 16)]
    b = [np64(t.cpu()) for t in run(x, 64)]
    for u, w in zip(a, b):
        assert rel_err(u, w) <= 2e-2


def test_training_workload_full_size_sampled():
    """B=4, H=16, n=8192, d=dv=128, decay 0.995: the whole batch runs on the GPU; heads
    (b=0, h=0), (b=1, h=7), (b=3, h=15) are compared with the oracle."""
    w = inputs.WORKLOADS["train"]
    x = inputs.make(w, device="cuda")
    g = x["gamma"].cuda()
    dq, dk, dv = hla.backward(x["q"], x["k"], x["v"], x["dout"], gamma=g, chunk=w.chunk)
    for b, h in ((0, 0), (1, 7), (3, 15)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = cref.backward(np32(x["q"][sl]), np32(x["k"][sl]), np32(x["v"][sl]), np32(x["dout"][sl]),
                            x["gamma"][h:h + 1].double().numpy())
        for name, gg, rr in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            assert rel_err(np64(gg[sl].cpu()), rr) <= 2e-2, (name, b, h)


def test_unsupported_variants_are_reported():
    x = inputs.make_custom(1, 1, 32, 16, 32, torch.bfloat16, seed=5, with_dout=True)
    with pytest.raises(HLA2Error):  # the bf16 tensor-core backward needs d == dv
        run(x, 16)


@pytest.mark.parametrize("d, dv", [(16, 16), (32, 64), (64, 32), (64, 64), (128, 128), (16, 128)])
@pytest.mark.parametrize("chunk", [16, 32, 64])
def test_fp32_gradients_match_oracle(d, dv, chunk):
    """float32 inputs: the SIMT reverse-mode kernels, several chunks and a ragged tail."""
    n = 3 * chunk + 7
    x = inputs.make_custom(1, 2, n, d, dv, torch.float32, seed=d + 3 * dv + chunk, gamma=(0.9, 0.999), with_dout=True)
    got = run(x, chunk)
    for name, gg, rr in zip(("dq", "dk", "dv"), got, oracle(x)):
        assert rel_err(np64(gg.cpu()), rr) <= 1e-4, name


@pytest.mark.parametrize("n", [1, 31, 33, 700, 3000])
def test_fp32_lengths_and_segments(n):
    """float32 gradients across many segments (the reverse scan and its cross term at 1e-4)."""
    x = inputs.make_custom(1, 3, n, 32, 32, torch.float32, seed=n + 11, gamma=(0.99, 0.9999), with_dout=True)
    got = run(x, 32)
    for name, gg, rr in zip(("dq", "dk", "dv"), got, oracle(x)):
        assert rel_err(np64(gg.cpu()), rr) <= 1e-4, (name, n)


def test_fp32_segments_of_several_chunks():
    """152 heads of 1024 tokens at width 32: the float32 forward and reverse passes run 4
    segments of 8 chunks per head, so the states move from chunk to chunk within a segment."""
    x = inputs.make_custom(8, 19, 1024, 64, 64, torch.float32, seed=13, gamma=(0.9, 0.999), with_dout=True)
    nseg, seg_chunks, _ = hla.forward_plan(8, 19, 1024, 64, 64, 32, dtype=torch.float32)
    assert seg_chunks >= 4 and nseg >= 2
    g = x["gamma"].cuda()
    o = hla.forward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), gamma=g, chunk=32)
    ref_o = cref.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), x["gamma"].double().numpy())
    assert rel_err(np64(o.cpu()), ref_o) <= 1e-4
    got = run(x, 32)
    for name, gg, rr in zip(("dq", "dk", "dv"), got, oracle(x)):
        assert rel_err(np64(gg.cpu()), rr) <= 1e-4, name


def test_fp32_no_decay_and_host_tensors():
    x = inputs.make_custom(2, 1, 300, 16, 32, torch.float32, seed=12, gamma=None, with_dout=True)
    got = hla.backward(x["q"], x["k"], x["v"], x["dout"], chunk=16)  # CPU tensors in and out
    assert got[0].device.type == "cpu"
    for name, gg, rr in zip(("dq", "dk", "dv"), got, oracle(x)):
        assert rel_err(np64(gg), rr) <= 1e-4, name


@pytest.mark.parametrize("B,H,n,d", [(1, 3, 333, 64), (2, 2, 2000, 64), (1, 4, 1000, 128), (4, 16, 300, 32)])
def test_training_forward_saves_for_backward(B, H, n, d):
    """forward(save_for_backward=True) writes the same output as the oracle, and
    backward(saved=...) returns the gradients of a backward that recomputes the forward,
    bit for bit (the same kernels on the same segmentation)."""
    x = inputs.make_custom(B, H, n, d, d, torch.bfloat16, seed=n + d, gamma=(0.95, 0.999), with_dout=True)
    q, k, v, do = (x[t].cuda() for t in ("q", "k", "v", "dout"))
    g = x["gamma"].cuda()
    o, saved = hla.forward(q, k, v, gamma=g, chunk=64, save_for_backward=True)
    ref_o = cref.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), x["gamma"].double().numpy())
    assert rel_err(np64(o.cpu()), ref_o) <= 2e-2
    fresh = hla.backward(q, k, v, do, gamma=g, chunk=64)
    reused = hla.backward(q, k, v, do, gamma=g, chunk=64, saved=saved)
    for a, b in zip(fresh, reused):
        assert torch.equal(a, b)
    ref = oracle(x)
    for gg, rr in zip(reused, ref):
        assert rel_err(np64(gg.cpu()), rr) <= 2e-2


def test_save_for_backward_rejects_uncovered_requests():
    x = inputs.make_custom(1, 2, 100, 64, 64, torch.bfloat16, seed=5, gamma=0.99)
    q, k, v = (x[t].cuda() for t in ("q", "k", "v"))
    with pytest.raises(HLA2Error):
        hla.forward(q, k, v, gamma=x["gamma"].cuda(), normalize=True, save_for_backward=True)
    _, saved = hla.forward(q, k, v, gamma=x["gamma"].cuda(), chunk=64, save_for_backward=True)
    with pytest.raises(ValueError):  # other chunk than the saving forward
        hla.backward(q, k, v, v, gamma=x["gamma"].cuda(), chunk=32, saved=saved)


def _normalized_reference(x, eps):
    """Oracle gradients of the normalised output and the conditioning of their quotient-rule
    split: kappa = (max|numerator part| + max|denominator part|) / max|sum|, per gradient."""
    q, k, v, do = (np32(x[t]) for t in ("q", "k", "v", "dout"))
    g = x["gamma"].double().numpy()
    ones = np.ones(v.shape[:-1] + (1,), dtype=np.float32)
    num = cref.forward(q, k, v, g)
    den = cref.forward(q, k, ones, g)[..., 0]
    inv = 1.0 / (den + eps)
    p1 = cref.backward(q, k, v, do * inv[..., None], g)
    p2 = cref.backward(q, k, ones, (-np.sum(do * num, axis=-1) * inv * inv)[..., None], g)
    ref = cref.backward_normalized(q, k, v, do, g, eps)
    kappa = [(np.abs(a).max() + np.abs(b).max()) / np.abs(a + b).max() for a, b in zip(p1[:2], p2[:2])] + [1.0]
    return ref, kappa


@pytest.mark.parametrize("d,chunk,n", [(32, 32, 300), (64, 64, 1000), (64, 128, 777), (128, 64, 400)])
def test_normalized_gradients_match_oracle(d, chunk, n):
    """Ratio-normalised backward (quotient rule over unnormalised passes) against the oracle's
    normalised adjoint on the normalised workload's recipe (positive q, k: den > 0).

    dq and dk are a difference of a numerator part and a denominator part that can be many
    times larger than the result (kappa, the parts' magnitude over the result's, reaches
    tens here).  The library therefore runs the composition in float32, and the bf16 bar
    of 2e-2 holds whatever kappa is."""
    x = inputs.make_custom(2, 2, n, d, d, torch.bfloat16, seed=40 + d + n, qk="softplus", v_scale="unit",
                           gamma=(0.95, 0.999), with_dout=True)
    g = x["gamma"].cuda()
    got = hla.backward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["dout"].cuda(), gamma=g, chunk=chunk,
                       normalize=True, eps=1e-6)
    ref, kappa = _normalized_reference(x, 1e-6)
    for name, gg, rr, kk in zip(("dq", "dk", "dv"), got, ref, kappa):
        assert torch.isfinite(gg.float()).all(), name
        assert rel_err(np64(gg.cpu()), rr) <= 2e-2, (name, kk)


@pytest.mark.parametrize("d, dv, chunk", [(32, 32, 32), (64, 16, 64), (16, 64, 16)])
def test_normalized_gradients_fp32(d, dv, chunk):
    """float32 inputs: the normalised gradients at the float32 bar, 1e-4."""
    x = inputs.make_custom(1, 2, 333, d, dv, torch.float32, seed=60 + d + dv, qk="softplus", v_scale="unit",
                           gamma=(0.95, 0.999), with_dout=True)
    got = hla.backward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["dout"].cuda(), gamma=x["gamma"].cuda(),
                       chunk=chunk, normalize=True, eps=1e-6)
    ref, kappa = _normalized_reference(x, 1e-6)
    for name, gg, rr, kk in zip(("dq", "dk", "dv"), got, ref, kappa):
        assert rel_err(np64(gg.cpu()), rr) <= 1e-4, (name, kk)


@pytest.mark.parametrize("d", [32, 64, 128])
def test_normalized_gradients_short_memory(d):
    """Positive q, k scaled by 1/sqrt(d) and a short memory (decay 0.8-0.9), at 2e-2."""
    x = inputs.make_custom(1, 3, 500, d, d, torch.bfloat16, seed=50 + d, qk="softplus", v_scale="unit",
                           gamma=(0.8, 0.9), with_dout=True)
    x["q"] = (x["q"].float() / d ** 0.5).to(torch.bfloat16)
    x["k"] = (x["k"].float() / d ** 0.5).to(torch.bfloat16)
    ref, kappa = _normalized_reference(x, 1e-6)
    got = hla.backward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["dout"].cuda(), gamma=x["gamma"].cuda(),
                       chunk=64, normalize=True, eps=1e-6)
    for name, gg, rr, kk in zip(("dq", "dk", "dv"), got, ref, kappa):
        assert rel_err(np64(gg.cpu()), rr) <= 2e-2, (name, kk)


def test_normalized_workload_gradients():
    """The normalised workload itself (B=2 H=8 n=2048 d=dv=64 bf16, chunk 64): the float32 passes
    run 16 segments of 4 chunks per head."""
    import dataclasses

    w = dataclasses.replace(inputs.WORKLOADS["normed"], with_dout=True)
    x = inputs.make(w, seed=w.seed)
    got = hla.backward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["dout"].cuda(), gamma=x["gamma"].cuda(),
                       chunk=w.chunk, normalize=True, eps=w.eps)
    ref, kappa = _normalized_reference(x, w.eps)
    for name, gg, rr, kk in zip(("dq", "dk", "dv"), got, ref, kappa):
        assert rel_err(np64(gg.cpu()), rr) <= 2e-2, (name, kk)


def test_normalized_gradients_bf16_unequal_dims():
    """The normalised backward composes float32 passes, so bf16 d != dv works too."""
    x = inputs.make_custom(1, 2, 260, 64, 32, torch.bfloat16, seed=77, qk="softplus", v_scale="unit",
                           gamma=(0.95, 0.999), with_dout=True)
    got = hla.backward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["dout"].cuda(), gamma=x["gamma"].cuda(),
                       chunk=32, normalize=True, eps=1e-6)
    ref, kappa = _normalized_reference(x, 1e-6)
    for name, gg, rr, kk in zip(("dq", "dk", "dv"), got, ref, kappa):
        assert rel_err(np64(gg.cpu()), rr) <= 2e-2, (name, kk)
