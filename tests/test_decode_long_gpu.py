"""The streaming-decode workload at its stated length, through the C ABI.

256 sequences x 32 heads, d = dv = 128: a 4096-token bf16 prefill (decay 0.999) through the
forward's final state, then all 1024 single-token decode steps with fresh seeded q, k, v.
Sequences 0..3 (128 heads) are followed by the float64 oracle over the same prefill and
steps: the outputs are compared at every 64th step and at the last, and the state after the
last step part by part (S, C, m, G, h), so that float32 drift of the state over 1024 steps
against float64 would show.  The same for the compact state and for multi-query sharing of
S (32 query heads in 8 key groups of 4).
"""
import numpy as np
import pytest
import torch

import chunked_scan_mixer_gb300 as hla
from chunked_scan_mixer_gb300 import inputs
from oracle import cref

from .helpers import assert_state_parts, np32, np64, rel_err

pytestmark = pytest.mark.gpu

SUB = slice(0, 4)  # sequences followed by the oracle


def _checked(step):
    return step % 64 == 63 or step == inputs.DECODE_STEPS - 1


def _prefill(w, group):
    """The workload's prefill on the GPU and on the oracle (sequences SUB).  With group > 1
    the keys and values of the first head of each group are shared by the group's heads."""
    x = inputs.make(w, device="cuda")
    if group > 1:
        for key in ("k", "v"):
            x[key] = x[key][:, ::group].repeat_interleave(group, dim=1).contiguous()
    g = x["gamma"].cuda()
    _, state = hla.forward(x["q"], x["k"], x["v"], gamma=g, chunk=w.chunk, return_final_state=True)
    gd = x["gamma"].double().numpy()
    _, st_ref = cref.forward(np32(x["q"][SUB]), np32(x["k"][SUB]), np32(x["v"][SUB]), gd, return_state=True)
    del x
    torch.cuda.synchronize()
    return state, st_ref, g, gd


@pytest.mark.parametrize("variant", ["packed", "compact", "multi_query"])
def test_decode_workload_all_steps(variant):
    w = inputs.WORKLOADS["decode_prefill"]
    N, H, d, dv = w.B, w.H, w.d, w.dv
    group = 4 if variant == "multi_query" else 1
    Hk = H // group
    state, st_ref, g, gd = _prefill(w, group)
    assert_state_parts(state[SUB].cpu().double().numpy(), st_ref, d, dv, 2e-2, "prefill")
    if variant == "compact":
        state = hla.state_to_compact(state, d, dv)
    elif variant == "multi_query":
        key_state, head_state = hla.mq_split_state(state, d, dv, group)
        del state
        gk = g[::group].contiguous()
    checked = 0
    for step in range(inputs.DECODE_STEPS):
        q, k, v = inputs.decode_step_inputs(step, N, H, d, dv, device="cuda")
        if variant == "multi_query":
            k, v = k[:, ::group].contiguous(), v[:, ::group].contiguous()
            o = hla.decode_step_mq(key_state, head_state, q, k, v, gamma=gk)
            k, v = k.repeat_interleave(group, dim=1), v.repeat_interleave(group, dim=1)
        else:
            o = hla.decode_step(state, q, k, v, gamma=g, compact=variant == "compact")
        ref = cref.decode_step(st_ref, np32(q[SUB]), np32(k[SUB]), np32(v[SUB]), gd)
        if _checked(step):
            assert rel_err(np64(o[SUB].cpu()), ref) <= 2e-2, step
            assert torch.isfinite(o.float()).all(), step
            checked += 1
    assert checked == inputs.DECODE_STEPS // 64 + (inputs.DECODE_STEPS % 64 != 0)
    if variant == "compact":
        state = hla.state_from_compact(state, d, dv)
    elif variant == "multi_query":
        state = hla.mq_merge_state(key_state[SUB], head_state[SUB], d, dv)
    assert_state_parts(state[SUB].cpu().double().numpy(), st_ref, d, dv, 2e-2, f"after {inputs.DECODE_STEPS} steps")
    assert Hk * group == H and np.isfinite(st_ref).all()
