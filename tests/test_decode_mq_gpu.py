"""GPU multi-query decode step (one key moment per group of query heads) against the float64
oracle, through the C ABI.

The oracle for a group is the single-head recurrence run on every head of the group with the
group's key and value (the equivalence is pinned in tests/test_oracle.py), so the reference
is the C oracle's decode on keys and values repeated over the heads."""
import numpy as np
import pytest
import torch

import chunked_scan_mixer_gb300 as hla
from chunked_scan_mixer_gb300 import inputs
from oracle import cref
from oracle import hla2_oracle as O

from .helpers import np32, np64, rel_err, tol_for

pytestmark = pytest.mark.gpu


def _prefill(N, Hk, group, d, dv, n, seed, gamma, qk="gauss"):
    """Oracle state after n tokens on keys and values shared within each group."""
    x = inputs.make_custom(N, Hk * group, n, d, dv, torch.float32, seed=seed, qk=qk)
    kx = inputs.make_custom(N, Hk, n, d, dv, torch.float32, seed=seed + 1, qk=qk)
    k = kx["k"].repeat_interleave(group, dim=1)
    v = kx["v"].repeat_interleave(group, dim=1)
    g = np.repeat(np.asarray(gamma, dtype=np.float64), group)
    _, st = cref.forward(np32(x["q"]), np32(k), np32(v), g, return_state=True)
    return st.astype(np.float32).astype(np.float64)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("d, dv", [(16, 16), (64, 64), (128, 128), (32, 64), (64, 32)])
@pytest.mark.parametrize("masked", [True, False])
def test_mq_decode_matches_oracle(dtype, group, d, dv, masked):
    N, Hk = 3, 2
    gamma = [0.95, 0.999]
    st = _prefill(N, Hk, group, d, dv, 30, seed=d + dv + group, gamma=gamma)
    key_state, head_state = hla.mq_split_state(torch.from_numpy(st).float().cuda(), d, dv, group)
    ref_state = st.copy()
    gk = torch.tensor(gamma, dtype=torch.float32)
    for step in range(4):
        q, _, _ = inputs.decode_step_inputs(step, N, Hk * group, d, dv, dtype=dtype)
        _, k, v = inputs.decode_step_inputs(100 + step, N, Hk, d, dv, dtype=dtype)
        o = hla.decode_step_mq(key_state, head_state, q.cuda(), k.cuda(), v.cuda(), gamma=gk.cuda(), masked=masked)
        ref = cref.decode_step(ref_state, np32(q), np32(k.repeat_interleave(group, dim=1)),
                               np32(v.repeat_interleave(group, dim=1)), np.repeat(gamma, group), masked=masked)
        assert rel_err(np64(o.cpu()), ref) <= tol_for(dtype), step
    got = O.unpack_state(hla.mq_merge_state(key_state, head_state, d, dv).cpu().double().numpy(), d, dv)
    want = O.unpack_state(ref_state, d, dv)
    keys = ("S", "C", "m", "G", "h") if masked else ("S", "C", "m")
    for key in keys:
        assert rel_err(got[key], want[key]) <= 1e-5, key


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_mq_decode_normalized(dtype):
    N, Hk, group, d = 2, 2, 4, 64
    gamma = [0.97, 0.995]
    st = _prefill(N, Hk, group, d, d, 12, seed=77, gamma=gamma, qk="softplus")
    key_state, head_state = hla.mq_split_state(torch.from_numpy(st).float().cuda(), d, d, group)
    ref_state = st.copy()
    for step in range(3):
        q, _, _ = inputs.decode_step_inputs(step, N, Hk * group, d, d, dtype=torch.float32)
        _, k, v = inputs.decode_step_inputs(200 + step, N, Hk, d, d, dtype=torch.float32)
        q, k, v = q.abs().to(dtype), k.abs().to(dtype), v.to(dtype)
        o = hla.decode_step_mq(key_state, head_state, q.cuda(), k.cuda(), v.cuda(), gamma=torch.tensor(gamma).cuda(),
                               normalize=True, eps=1e-6)
        ref = cref.decode_step(ref_state, np32(q), np32(k.repeat_interleave(group, dim=1)),
                               np32(v.repeat_interleave(group, dim=1)), np.repeat(gamma, group), normalize=True,
                               eps=1e-6)
        assert rel_err(np64(o.cpu()), ref) <= tol_for(dtype), step


def test_mq_equals_single_head_step_on_repeated_keys():
    """The multi-query step and the per-head step on repeated keys, values and S give the
    same outputs and states (fp32, same kernel arithmetic order within a pass)."""
    N, Hk, group, d, dv = 4, 3, 4, 128, 128
    st = _prefill(N, Hk, group, d, dv, 20, seed=88, gamma=[0.99, 0.995, 0.999])
    full = torch.from_numpy(st).float().cuda()
    key_state, head_state = hla.mq_split_state(full, d, dv, group)
    gam = torch.tensor([0.99, 0.995, 0.999])
    q, _, _ = inputs.decode_step_inputs(9, N, Hk * group, d, dv, dtype=torch.bfloat16)
    _, k, v = inputs.decode_step_inputs(19, N, Hk, d, dv, dtype=torch.bfloat16)
    o_mq = hla.decode_step_mq(key_state, head_state, q.cuda(), k.cuda(), v.cuda(), gamma=gam.cuda())
    o_1 = hla.decode_step(full, q.cuda(), k.repeat_interleave(group, dim=1).cuda(),
                          v.repeat_interleave(group, dim=1).cuda(), gamma=gam.repeat_interleave(group).cuda())
    assert rel_err(np64(o_mq.cpu()), np64(o_1.cpu())) <= 2e-2
    merged = hla.mq_merge_state(key_state, head_state, d, dv)
    assert rel_err(merged.cpu().double().numpy(), full.cpu().double().numpy()) <= 1e-6


def test_mq_decode_full_width_sampled():
    """The measured shape, 256 sequences x 32 query heads in 8 key groups at d = dv = 128:
    one step on a random state (S symmetric, as every sum of k k^T is), sampled heads
    against the oracle."""
    N, Hk, group, d, dv = 256, 8, 4, 128, 128
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    A = torch.randn((N, Hk, d, d), generator=gen, device="cuda") * 1e-2
    key_state = (0.5 * (A + A.transpose(-1, -2))).reshape(N, Hk, d * d).contiguous()
    del A
    head_state = torch.randn((N, Hk * group, hla.mq_head_state_floats(d, dv)), generator=gen, device="cuda") * 1e-2
    ks0, hs0 = key_state.clone(), head_state.clone()
    q, _, _ = inputs.decode_step_inputs(3, N, Hk * group, d, dv, dtype=torch.bfloat16, device="cuda")
    _, k, v = inputs.decode_step_inputs(13, N, Hk, d, dv, dtype=torch.bfloat16, device="cuda")
    gam = torch.linspace(0.99, 0.9999, Hk, device="cuda")
    o = hla.decode_step_mq(key_state, head_state, q, k, v, gamma=gam)
    torch.cuda.synchronize()
    for n_ in (0, 97, 255):
        for j in (0, 5, 7):
            heads = slice(j * group, (j + 1) * group)
            st = hla.mq_merge_state(ks0[n_:n_ + 1, j:j + 1], hs0[n_:n_ + 1, heads], d, dv).cpu().double().numpy()
            ref = cref.decode_step(st, np32(q[n_:n_ + 1, heads]),
                                   np32(k[n_:n_ + 1, j:j + 1].repeat_interleave(group, dim=1)),
                                   np32(v[n_:n_ + 1, j:j + 1].repeat_interleave(group, dim=1)),
                                   np.full(group, float(gam[j])))
            assert rel_err(np64(o[n_:n_ + 1, heads].cpu()), ref) <= 2e-2, (n_, j)
