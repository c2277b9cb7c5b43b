"""GPU decode step against the float64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import chunked_scan_mixer_gb300 as hla
from chunked_scan_mixer_gb300 import inputs
from oracle import cref
from oracle import hla2_oracle as O

from .helpers import assert_state_parts, np32, np64, rel_err, tol_for

pytestmark = pytest.mark.gpu


def prefill_state(N, H, d, dv, n, seed, gamma):
    """A realistic packed state: the oracle's final state after n random tokens."""
    x = inputs.make_custom(N, H, n, d, dv, torch.float32, seed=seed, gamma=gamma)
    g = None if x["gamma"] is None else x["gamma"].double().numpy()
    _, st = cref.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), g, return_state=True)
    return st, x["gamma"]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("d, dv", [(16, 16), (64, 64), (128, 128), (32, 64), (64, 32)])
@pytest.mark.parametrize("normalize", [False, True])
def test_decode_steps_match_oracle(dtype, d, dv, normalize):
    N, H = 3, 2
    st, gamma = prefill_state(N, H, d, dv, 40, seed=d + dv, gamma=(0.95, 0.999))
    if normalize:  # positive queries/keys keep the denominator away from zero
        st_q = inputs.make_custom(N, H, 6, d, dv, torch.float32, seed=99, qk="softplus", gamma=(0.95, 0.999))
        g = st_q["gamma"].double().numpy()
        _, st = cref.forward(np32(st_q["q"]), np32(st_q["k"]), np32(st_q["v"]), g, return_state=True)
    state_gpu = torch.from_numpy(st.astype(np.float32)).cuda()
    state_ref = st.astype(np.float32).astype(np.float64).copy()
    for step in range(5):
        q, k, v = inputs.decode_step_inputs(step, N, H, d, dv, dtype=dtype)
        if normalize:
            q, k = q.float().abs().to(dtype), k.float().abs().to(dtype)
        o = hla.decode_step(state_gpu, q.cuda(), k.cuda(), v.cuda(), gamma=gamma.cuda(),
                            normalize=normalize, eps=1e-6)
        ref = cref.decode_step(state_ref, np32(q), np32(k), np32(v), gamma.double().numpy(),
                               normalize=normalize, eps=1e-6)
        assert rel_err(np64(o.cpu()), ref) <= tol_for(dtype), step
    assert_state_parts(state_gpu.cpu().double().numpy(), state_ref, d, dv, 1e-5)


def test_decode_from_zero_equals_forward():
    N, H, d, n = 2, 3, 64, 37
    x = inputs.make_custom(N, H, n, d, d, torch.float32, seed=5, gamma=(0.9, 0.99))
    state = torch.zeros(N, H, hla.state_floats(d, d), device="cuda")
    outs = []
    for t in range(n):
        outs.append(hla.decode_step(state, x["q"][:, :, t].cuda(), x["k"][:, :, t].cuda(),
                                    x["v"][:, :, t].cuda(), gamma=x["gamma"].cuda()))
    o = torch.stack(outs, dim=2).cpu()
    ref, ref_state = cref.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), x["gamma"].double().numpy(),
                                  return_state=True)
    assert rel_err(np64(o), ref) <= 1e-4
    assert_state_parts(state.cpu().double().numpy(), ref_state, d, d, 1e-5)


def test_prefill_then_decode_matches_uninterrupted_oracle():
    """Checkpoint/resume: a GPU prefill's final state continues exactly like the oracle
    run over prefill + decode tokens."""
    N, H, d, n = 2, 4, 128, 300
    x = inputs.make_custom(N, H, n, d, d, torch.bfloat16, seed=6, gamma=0.999)
    _, fin = hla.forward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), gamma=x["gamma"].cuda(), chunk=64,
                         return_final_state=True)
    g = x["gamma"].double().numpy()
    _, ref_state = cref.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), g, return_state=True)
    assert_state_parts(fin.cpu().double().numpy(), ref_state, d, d, 2e-2, "prefill")
    state_ref = ref_state.copy()
    for step in range(4):
        q, k, v = inputs.decode_step_inputs(step, N, H, d, d)
        o = hla.decode_step(fin, q.cuda(), k.cuda(), v.cuda(), gamma=x["gamma"].cuda())
        ref = cref.decode_step(state_ref, np32(q), np32(k), np32(v), g)
        assert rel_err(np64(o.cpu()), ref) <= 2e-2
    assert_state_parts(fin.cpu().double().numpy(), state_ref, d, d, 2e-2, "after decode")


def test_decode_workload_full_width_sampled():
    """256 sequences x 32 heads, d = dv = 128: a 4096-token bf16 prefill through the
    forward (final state), then decode steps; sequences 0..3 (128 heads) are compared
    with the oracle run over the same tokens."""
    w = inputs.WORKLOADS["decode_prefill"]
    x = inputs.make(w, device="cuda")
    g = x["gamma"].cuda()
    _, state = hla.forward(x["q"], x["k"], x["v"], gamma=g, chunk=w.chunk, return_final_state=True)
    sub = slice(0, 4)
    gd = x["gamma"].double().numpy()
    _, st_ref = cref.forward(np32(x["q"][sub]), np32(x["k"][sub]), np32(x["v"][sub]), gd, return_state=True)
    del x
    assert_state_parts(state[sub].cpu().double().numpy(), st_ref, w.d, w.dv, 2e-2, "prefill")
    for step in range(3):
        q, k, v = inputs.decode_step_inputs(step, w.B, w.H, w.d, w.dv, device="cuda")
        o = hla.decode_step(state, q, k, v, gamma=g)
        ref = cref.decode_step(st_ref, np32(q[sub]), np32(k[sub]), np32(v[sub]), gd)
        assert rel_err(np64(o[sub].cpu()), ref) <= 2e-2, step
        assert torch.isfinite(o.float()).all()


@pytest.mark.parametrize("d, dv", [(16, 16), (64, 64), (128, 128), (32, 64)])
def test_compact_conversion_is_exact(d, dv):
    """To-compact keeps S's upper block triangle bit for bit (the oracle's own packing of the
    same layout); from-compact mirrors it back."""
    st, _ = prefill_state(2, 3, d, dv, 30, seed=70 + d, gamma=(0.95, 0.999))
    S = st[..., :d * d].reshape(2, 3, d, d)
    st = st.copy()
    st[..., :d * d] = (0.5 * (S + np.swapaxes(S, -1, -2))).reshape(2, 3, d * d)  # exactly symmetric
    full = torch.from_numpy(st.astype(np.float32)).cuda()
    c = hla.state_to_compact(full, d, dv)
    ref_c = O.compact_from_state(st.astype(np.float32).astype(np.float64), d, dv)
    assert np.array_equal(c.cpu().double().numpy(), ref_c)
    back = hla.state_from_compact(c, d, dv)
    assert torch.equal(back, full)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("d, dv", [(16, 16), (64, 64), (128, 128), (64, 32)])
@pytest.mark.parametrize("normalize", [False, True])
def test_compact_decode_matches_oracle(dtype, d, dv, normalize):
    """Decode steps on the compact state against the oracle's serial steps on the packed one."""
    N, H = 3, 2
    if normalize:
        xs = inputs.make_custom(N, H, 6, d, dv, torch.float32, seed=98, qk="softplus", gamma=(0.95, 0.999))
        gamma = xs["gamma"]
        _, st = cref.forward(np32(xs["q"]), np32(xs["k"]), np32(xs["v"]), gamma.double().numpy(), return_state=True)
    else:
        st, gamma = prefill_state(N, H, d, dv, 40, seed=d + dv + 1, gamma=(0.95, 0.999))
    st = st.astype(np.float32).astype(np.float64)
    state_gpu = hla.state_to_compact(torch.from_numpy(st.astype(np.float32)).cuda(), d, dv)
    # the oracle continues from the same S the compact state holds (its upper triangle)
    state_ref = O.state_from_compact(O.compact_from_state(st, d, dv), d, dv).copy()
    for step in range(5):
        q, k, v = inputs.decode_step_inputs(step, N, H, d, dv, dtype=dtype)
        if normalize:
            q, k = q.float().abs().to(dtype), k.float().abs().to(dtype)
        o = hla.decode_step(state_gpu, q.cuda(), k.cuda(), v.cuda(), gamma=gamma.cuda(), normalize=normalize,
                            eps=1e-6, compact=True)
        ref = cref.decode_step(state_ref, np32(q), np32(k), np32(v), gamma.double().numpy(), normalize=normalize,
                               eps=1e-6)
        assert rel_err(np64(o.cpu()), ref) <= tol_for(dtype), step
    got = hla.state_from_compact(state_gpu, d, dv).cpu().double().numpy()
    assert_state_parts(got, state_ref, d, dv, 1e-5)


def test_compact_decode_full_width_sampled():
    """Full decode width (256 sequences x 32 heads, d = dv = 128), compact state: sampled
    heads against the oracle."""
    N, H, d = 256, 32, 128
    gen = torch.Generator(device="cuda")
    gen.manual_seed(11)
    full = torch.randn((N, H, hla.state_floats(d, d)), generator=gen, device="cuda") * 1e-2
    S = full[..., :d * d].view(N, H, d, d)
    S.copy_(0.5 * (S + S.transpose(-1, -2)))
    c = hla.state_to_compact(full, d, d)
    g = torch.full((H,), 0.999, device="cuda")
    q, k, v = inputs.decode_step_inputs(0, N, H, d, d, device="cuda")
    o = hla.decode_step(c, q, k, v, gamma=g, compact=True)
    for (n_, h_) in ((0, 0), (17, 5), (255, 31), (128, 16)):
        st = full[n_:n_ + 1, h_:h_ + 1].double().cpu().numpy().copy()
        ref = cref.decode_step(st, np32(q[n_:n_ + 1, h_:h_ + 1].cpu()), np32(k[n_:n_ + 1, h_:h_ + 1].cpu()),
                               np32(v[n_:n_ + 1, h_:h_ + 1].cpu()), np.full(1, 0.999))
        assert rel_err(np64(o[n_:n_ + 1, h_:h_ + 1].cpu()), ref) <= 2e-2


def test_decode_step_captured_in_a_graph():
    """A serving loop's form of the step: one decode step captured in a CUDA graph and replayed
    with fresh q, k, v copied into the captured buffers gives, step by step, the eager step's
    outputs and state (bit for bit) and the oracle's."""
    N, H, d, dv = 4, 8, 128, 128
    st, gamma = prefill_state(N, H, d, dv, 40, seed=77, gamma=(0.95, 0.999))
    g = gamma.cuda()
    eager = torch.from_numpy(st.astype(np.float32)).cuda()
    state = eager.clone()
    state_ref = st.astype(np.float32).astype(np.float64).copy()
    qb, kb, vb = (torch.empty((N, H, x), dtype=torch.bfloat16, device="cuda") for x in (d, d, dv))
    out = torch.empty((N, H, dv), dtype=torch.bfloat16, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture, on a scratch copy of the state
        hla.decode_step(state.clone(), qb.zero_(), kb.zero_(), vb.zero_(), gamma=g, out=out)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        hla.decode_step(state, qb, kb, vb, gamma=g, out=out)
    for step in range(4):
        q, k, v = inputs.decode_step_inputs(100 + step, N, H, d, dv, dtype=torch.bfloat16)
        qb.copy_(q)
        kb.copy_(k)
        vb.copy_(v)
        graph.replay()
        o_eager = hla.decode_step(eager, q.cuda(), k.cuda(), v.cuda(), gamma=g)
        torch.cuda.synchronize()
        assert torch.equal(out, o_eager), step
        assert torch.equal(state, eager), step
        ref = cref.decode_step(state_ref, np32(q), np32(k), np32(v), gamma.double().numpy())
        assert rel_err(np64(out.cpu()), ref) <= tol_for(torch.bfloat16), step
