"""GPU unmasked output (o_t = q_t^T S_t C_t, HLA2_FLAG_UNMASKED) against the float64 oracle,
through the C ABI: forward on the fp32 and tensor-core paths, the scan of the unmasked
monoid across segments, normalisation, state in and out, and the decode step.

Bars as for the masked output: max|gpu - oracle| / max|oracle| <= 1e-4 for float32 inputs
and <= 2e-2 for bf16 inputs."""
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
    return hla.forward(q, k, v, gamma=None if x["gamma"] is None else x["gamma"].cuda(), masked=False, **kw)


def oracle(x, normalize=False, eps=1e-6, init_state=None, return_state=False):
    g = None if x["gamma"] is None else x["gamma"].double().numpy()
    return cref.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), g, normalize=normalize, eps=eps,
                        init_state=init_state, return_state=return_state, masked=False)


def test_tiny_fp32_against_brute_force():
    x = inputs.make_custom(1, 2, 40, 16, 16, torch.float32, seed=50, gamma=(0.9, 1.0))
    o = run_gpu(x, chunk=16).cpu()
    ref = O.brute_force_forward(np64(x["q"]), np64(x["k"]), np64(x["v"]), x["gamma"].double().numpy(),
                                masked=False)
    assert rel_err(np64(o), ref) <= 1e-4
    assert rel_err(np64(o), oracle(x)) <= 1e-4
    # and it is not the masked output
    masked = hla.forward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), gamma=x["gamma"].cuda(), chunk=16).cpu()
    assert rel_err(np64(masked), ref) > 1e-2


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("chunk", [16, 32, 64, 128])
def test_bf16_shapes_and_chunks(d, chunk):
    # d = 128 at chunk 128 has no kernel (its tiles exceed one CTA's shared memory) and runs
    # at the widest narrower width that has one
    n = 3 * chunk + 5  # several chunks and a ragged tail
    x = inputs.make_custom(2, 3, n, d, d, torch.bfloat16, seed=d + chunk + 1, gamma=(0.9, 1.0))
    o = run_gpu(x, chunk=chunk).cpu()
    assert rel_err(np64(o), oracle(x)) <= 2e-2


@pytest.mark.parametrize("d, dv", [(16, 16), (32, 32), (64, 64), (32, 64), (64, 16)])
@pytest.mark.parametrize("chunk", [16, 32])
def test_fp32_shapes(d, dv, chunk):
    n = 4 * chunk + 3
    x = inputs.make_custom(1, 2, n, d, dv, torch.float32, seed=7 * d + dv + 1, gamma=(0.95, 0.999))
    o = run_gpu(x, chunk=chunk).cpu()
    assert rel_err(np64(o), oracle(x)) <= 1e-4


def test_bf16_unequal_dims_use_simt_path():
    x = inputs.make_custom(1, 2, 200, 32, 64, torch.bfloat16, seed=51, gamma=0.97)
    o = run_gpu(x, chunk=32).cpu()
    assert rel_err(np64(o), oracle(x)) <= 2e-2


@pytest.mark.parametrize("n", [1, 2, 17, 64, 65, 1000])
def test_ragged_and_short_sequences(n):
    x = inputs.make_custom(1, 2, n, 64, 64, torch.bfloat16, seed=n + 3, gamma=(0.9, 0.99))
    o = run_gpu(x, chunk=64).cpu()
    assert rel_err(np64(o), oracle(x)) <= 2e-2


def test_many_segments_long_sequence_fp32():
    """The unmasked monoid's inter-segment scan (decayed prefixes of S and C) at 1e-4."""
    x = inputs.make_custom(1, 1, 4096, 16, 16, torch.float32, seed=52, gamma=0.999)
    o = run_gpu(x, chunk=16).cpu()
    assert rel_err(np64(o), oracle(x)) <= 1e-4


def test_long_context_shapes_bf16():
    """B=1 H=16 n=65536 d=dv=64 at chunk 128 (the tcgen05 stored-p kernels, unmasked variant),
    every output compared, per head."""
    x = inputs.make("long")
    o = run_gpu(x, chunk=x["chunk"]).cpu()
    ref = oracle(x)
    for h in range(16):
        assert rel_err(np64(o[0, h]), ref[0, h]) <= 2e-2, h


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_normalized_with_decay(dtype):
    x = inputs.make_custom(2, 2, 300, 32, 32, dtype, seed=53, qk="softplus", v_scale="unit",
                           gamma=(0.95, 0.999))
    o = run_gpu(x, chunk=32, normalize=True, eps=1e-6).cpu()
    assert rel_err(np64(o), oracle(x, normalize=True)) <= tol_for(dtype)


@pytest.mark.parametrize("dtype, d", [(torch.float32, 16), (torch.bfloat16, 64), (torch.bfloat16, 128)])
def test_final_state_matches_oracle(dtype, d):
    """S, C, m after the last token; G and h are not tracked and come back as 0."""
    x = inputs.make_custom(1, 2, 5 * 64 + 9, d, d, dtype, seed=54, gamma=(0.97, 0.999))
    o, fin = run_gpu(x, chunk=64 if d > 16 else 16, return_final_state=True)
    ref, ref_state = oracle(x, return_state=True)
    assert rel_err(np64(o.cpu()), ref) <= tol_for(dtype)
    got = O.unpack_state(np64(fin.cpu()), d, d)
    want = O.unpack_state(ref_state, d, d)
    for key in ("S", "C", "m"):
        assert rel_err(got[key], want[key]) <= tol_for(dtype), key
    assert not got["G"].any() and not got["h"].any()


@pytest.mark.parametrize("dtype, d", [(torch.float32, 32), (torch.bfloat16, 64)])
def test_continuation_from_init_state(dtype, d):
    """Unmasked forward over [0, n) equals [0, m) then [m, n) from its final state."""
    x = inputs.make_custom(2, 2, 700, d, d, dtype, seed=55, gamma=(0.99, 0.999))
    m = 300
    first = {key: (val[:, :, :m].contiguous() if key in ("q", "k", "v") else val) for key, val in x.items()}
    second = {key: (val[:, :, m:].contiguous() if key in ("q", "k", "v") else val) for key, val in x.items()}
    _, s1 = run_gpu(first, chunk=32, return_final_state=True)
    o2 = run_gpu(second, chunk=32, init_state=s1).cpu()
    assert rel_err(np64(o2), oracle(x)[:, :, m:]) <= tol_for(dtype)


def test_init_state_cross_summaries_are_ignored():
    """The unmasked output reads S, C, m of init_state only: G and h may hold anything."""
    x = inputs.make_custom(1, 2, 150, 32, 32, torch.float32, seed=56, gamma=0.98)
    r = np.random.default_rng(57)
    init = r.standard_normal((1, 2, O.state_floats(32, 32))) * 0.1
    o1 = run_gpu(x, chunk=32, init_state=torch.from_numpy(init).float().cuda()).cpu()
    junk = O.unpack_state(init, 32, 32)
    junk["G"] = junk["G"] + 5.0
    junk["h"] = junk["h"] - 3.0
    o2 = run_gpu(x, chunk=32, init_state=torch.from_numpy(O.pack_state(junk)).float().cuda()).cpu()
    assert torch.equal(o1, o2)
    ref = oracle(x, init_state=init.astype(np.float32).astype(np.float64))
    assert rel_err(np64(o1), ref) <= 1e-4


def test_empty_sequence_zeroes_cross_summaries():
    x = inputs.make_custom(1, 2, 0, 16, 16, torch.float32, seed=58, gamma=0.9)
    init = torch.randn(1, 2, hla.state_floats(16, 16))
    o, fin = run_gpu(x, chunk=16, init_state=init.cuda(), return_final_state=True)
    got = O.unpack_state(np64(fin.cpu()), 16, 16)
    want = O.unpack_state(np64(init), 16, 16)
    for key in ("S", "C", "m"):
        assert np.array_equal(got[key], want[key])
    assert not got["G"].any() and not got["h"].any()


def test_causality_on_gpu():
    x = inputs.make_custom(1, 2, 500, 64, 64, torch.bfloat16, seed=59, gamma=0.99)
    o1 = run_gpu(x, chunk=64).cpu()
    y = {key: (val.clone() if key in ("q", "k", "v") else val) for key, val in x.items()}
    y["q"][:, :, 300:] = torch.randn_like(y["q"][:, :, 300:].float()).to(torch.bfloat16)
    y["v"][:, :, 300:] = 0
    o2 = run_gpu(y, chunk=64).cpu()
    assert torch.equal(o1[:, :, :300], o2[:, :, :300])


def test_host_tensors_pipelined():
    x = inputs.make_custom(2, 8, 1000, 64, 64, torch.bfloat16, seed=60, gamma=0.995)
    o = hla.forward(x["q"].pin_memory(), x["k"].pin_memory(), x["v"].pin_memory(), gamma=x["gamma"],
                    chunk=64, masked=False)
    assert o.device.type == "cpu"
    assert rel_err(np64(o), oracle(x)) <= 2e-2


def test_save_for_backward_is_refused():
    x = inputs.make_custom(1, 1, 64, 64, 64, torch.bfloat16, seed=61, gamma=0.99)
    with pytest.raises(hla.HLA2Error):
        run_gpu(x, chunk=64, save_for_backward=True)


# ---- decode ---------------------------------------------------------------------------------

@pytest.mark.parametrize("compact", [False, True])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("d, dv", [(16, 16), (64, 64), (128, 128), (32, 64)])
@pytest.mark.parametrize("normalize", [False, True])
def test_decode_steps_match_oracle(compact, dtype, d, dv, normalize):
    N, H = 3, 2
    qk = "softplus" if normalize else "gauss"
    pre = inputs.make_custom(N, H, 40, d, dv, torch.float32, seed=d + dv + 5, qk=qk, gamma=(0.95, 0.999))
    g = pre["gamma"].double().numpy()
    _, st = cref.forward(np32(pre["q"]), np32(pre["k"]), np32(pre["v"]), g, return_state=True)
    st = st.astype(np.float32).astype(np.float64)
    state_ref = st.copy()
    state_gpu = torch.from_numpy(st).float().cuda()
    if compact:
        state_gpu = hla.state_to_compact(state_gpu, d, dv)
    G0 = O.unpack_state(st, d, dv)["G"].copy()
    for step in range(5):
        q, k, v = inputs.decode_step_inputs(step, N, H, d, dv, dtype=dtype)
        if normalize:
            q, k = q.float().abs().to(dtype), k.float().abs().to(dtype)
        o = hla.decode_step(state_gpu, q.cuda(), k.cuda(), v.cuda(), gamma=pre["gamma"].cuda(),
                            normalize=normalize, eps=1e-6, compact=compact, masked=False)
        ref = cref.decode_step(state_ref, np32(q), np32(k), np32(v), g, normalize=normalize, eps=1e-6,
                               masked=False)
        assert rel_err(np64(o.cpu()), ref) <= tol_for(dtype), step
    full = hla.state_from_compact(state_gpu, d, dv) if compact else state_gpu
    got = O.unpack_state(full.cpu().double().numpy(), d, dv)
    want = O.unpack_state(state_ref, d, dv)
    for key in ("S", "C", "m"):
        assert rel_err(got[key], want[key]) <= 1e-5, key
    assert np.array_equal(got["G"], G0)  # G and h untouched


def test_prefill_then_decode_matches_oracle():
    """Unmasked GPU prefill (final state) continued by unmasked decode steps equals the
    oracle's unmasked output over all the tokens."""
    N, H, d, n0, steps = 2, 4, 64, 300, 6
    x = inputs.make_custom(N, H, n0 + steps, d, d, torch.bfloat16, seed=62, gamma=(0.99, 0.995, 0.999, 1.0))
    pre = {key: (val[:, :, :n0].contiguous() if key in ("q", "k", "v") else val) for key, val in x.items()}
    _, state = run_gpu(pre, chunk=64, return_final_state=True)
    outs = []
    for t in range(n0, n0 + steps):
        outs.append(hla.decode_step(state, x["q"][:, :, t].cuda(), x["k"][:, :, t].cuda(), x["v"][:, :, t].cuda(),
                                    gamma=x["gamma"].cuda(), masked=False))
    o = torch.stack(outs, dim=2).cpu()
    assert rel_err(np64(o), oracle(x)[:, :, n0:]) <= 2e-2


# ---- the tcgen05 path (bf16, d = dv = 64, chunk 128, unnormalised) ----------------------------

def _run_kernel(x, kernel=None):
    import os

    old = os.environ.pop("HLA2_KERNEL", None)
    if kernel:
        os.environ["HLA2_KERNEL"] = kernel
    try:
        o = run_gpu(x, chunk=128)
        hla.check_status()
        return o.cpu()
    finally:
        os.environ.pop("HLA2_KERNEL", None)
        if old is not None:
            os.environ["HLA2_KERNEL"] = old


@pytest.mark.parametrize("n", [1, 127, 128, 129, 1000, 128 * 40, 4096 + 33])
def test_tcgen05_path_lengths(n):
    x = inputs.make_custom(1, 3, n, 64, 64, torch.bfloat16, seed=n + 70, gamma=(0.97, 0.9999))
    o = _run_kernel(x)
    assert rel_err(np64(o), oracle(x)) <= 2e-2


def test_tcgen05_and_mma_paths_agree():
    """Unmasked output of the tcgen05 kernels and of the mma.sync kernels on the same inputs
    (many heads, multi-chunk segments)."""
    x = inputs.make_custom(2, 8, 128 * 24 + 5, 64, 64, torch.bfloat16, seed=71, gamma=(0.99, 0.9999))
    a = _run_kernel(x)
    b = _run_kernel(x, "mma")
    ref = oracle(x)
    assert rel_err(np64(a), ref) <= 2e-2
    assert rel_err(np64(b), ref) <= 2e-2
    assert rel_err(np64(a), np64(b)) <= 2e-2


@pytest.mark.parametrize("gamma", [None, (0.5, 0.9)])
def test_tcgen05_multi_chunk_segments_decay_extremes(gamma):
    """The unmasked output on segments of several chunks (the stored-p kernels), without decay
    and with strong decay, where the carry's share g^(it W + r + 1) underflows to zero."""
    B, H, n = 1, 16, 128 * 40 + 9
    nseg, seg_chunks, _ = hla.forward_plan(B, H, n, 64, 64, 128)
    assert nseg > 1 and seg_chunks >= 2
    x = inputs.make_custom(B, H, n, 64, 64, torch.bfloat16, seed=32, gamma=gamma)
    o = _run_kernel(x)
    assert torch.isfinite(o.float()).all()
    assert rel_err(np64(o), oracle(x)) <= 2e-2


@pytest.mark.parametrize("B,H,n", [(1, 16, 128 * 40 + 9), (2, 8, 100)])
def test_tcgen05_final_state(B, H, n):
    """The unmasked final state from the tcgen05 path (chunk 128): S, C, m against the oracle on
    multi-segment and one-segment calls; G and h are not tracked and come back as 0."""
    x = inputs.make_custom(B, H, n, 64, 64, torch.bfloat16, seed=55 + H, gamma=(0.97, 0.9999))
    o, fin = run_gpu(x, chunk=128, return_final_state=True)
    hla.check_status()
    ref, ref_state = oracle(x, return_state=True)
    assert rel_err(np64(o.cpu()), ref) <= 2e-2
    got = O.unpack_state(np64(fin.cpu()), 64, 64)
    want = O.unpack_state(ref_state, 64, 64)
    for key in ("S", "C", "m"):
        assert rel_err(got[key], want[key]) <= 2e-2, key
    assert not got["G"].any() and not got["h"].any()


def test_tcgen05_prefill_from_state_then_decode():
    """Unmasked prefill at chunk 128 from a carried-in state, then decode steps, against the
    oracle over the whole sequence."""
    B, H, m, n2, steps = 1, 16, 300, 128 * 40 + 9, 3
    x = inputs.make_custom(B, H, m + n2 + steps, 64, 64, torch.bfloat16, seed=57, gamma=(0.98, 0.9999))
    g = x["gamma"].cuda()
    part = lambda lo, hi: [x[t][:, :, lo:hi].contiguous().cuda() for t in ("q", "k", "v")]
    _, s1 = hla.forward(*part(0, m), gamma=g, chunk=32, return_final_state=True, masked=False)
    o2, s2 = hla.forward(*part(m, m + n2), gamma=g, chunk=128, init_state=s1, return_final_state=True,
                         masked=False)
    hla.check_status()
    ref = oracle(x)
    assert rel_err(np64(o2.cpu()), ref[:, :, m:m + n2]) <= 2e-2
    for t in range(m + n2, m + n2 + steps):
        q, k, v = part(t, t + 1)
        o = hla.decode_step(s2, q[:, :, 0], k[:, :, 0], v[:, :, 0], gamma=g, masked=False)
        assert rel_err(np64(o.cpu()), ref[:, :, t]) <= 2e-2, t
