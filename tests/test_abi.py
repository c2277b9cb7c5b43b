"""C-ABI checks that need no GPU: the library loads, exports every function the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes

import pytest
import torch

import chunked_scan_mixer_gb300 as hla
from chunked_scan_mixer_gb300.hla2 import EXPORTED_SYMBOLS, Opts

from .helpers import header_functions


@pytest.fixture(scope="module")
def L():
    return hla.lib()


def test_exports_every_declared_function(L):
    declared = header_functions()
    assert declared, "no declarations parsed from include/hla2.h"
    for name in declared:
        assert hasattr(L, name), f"{name} declared in hla2.h but not exported"
    assert set(declared) == set(EXPORTED_SYMBOLS)


def test_version_and_sizes(L):
    assert L.hla2_version() >= 100
    assert hla.state_floats(128, 128) == 128 * 128 + 2 * 128 * 128 + 2 * 128
    assert hla.state_floats(16, 32) == 16 * 16 + 2 * 16 * 32 + 2 * 16


def _fwd(L, **kw):
    # distinct (never dereferenced) addresses: every check below runs before any launch
    args = dict(q=ctypes.c_void_p(0x10000), k=ctypes.c_void_p(0x20000), v=ctypes.c_void_p(0x30000),
                out=ctypes.c_void_p(0x40000), B=1, H=1, n=16, d=16, dv=16, gamma=None, normalize=0,
                chunk=16, stream=None, opts=Opts(1, 1e-6, None, 0, None, None))
    args.update(kw)
    o = args.pop("opts")
    rc = L.hla2_forward(args["q"], args["k"], args["v"], args["out"], args["B"], args["H"], args["n"],
                        args["d"], args["dv"], args["gamma"], args["normalize"], args["chunk"],
                        args["stream"], None if o is None else ctypes.byref(o))
    return rc, L.hla2_last_error().decode()


@pytest.mark.parametrize("kw, code", [
    (dict(opts=None), -1),
    (dict(d=48), -1),
    (dict(dv=8), -1),
    (dict(chunk=24), -1),
    (dict(n=-1), -1),
    (dict(normalize=2), -1),
    (dict(opts=Opts(7, 1e-6, None, 0, None, None)), -1),
    (dict(q=None), -1),
    (dict(k=ctypes.c_void_p(18)), -1),
    (dict(out=ctypes.c_void_p(0x10000)), -1),         # out is q
    (dict(out=ctypes.c_void_p(0x30000 + 256)), -1),   # out overlaps the end of v (16 x 16 bf16)
    (dict(), -3),  # no workspace
])
def test_forward_rejects_bad_arguments(L, kw, code):
    rc, msg = _fwd(L, **kw)
    assert rc == code, msg
    assert msg


def test_forward_adjacent_out_is_accepted(L):
    # out right after v (16 x 16 bf16 = 512 bytes): no overlap, so the call gets as far as the
    # workspace check
    rc, msg = _fwd(L, out=ctypes.c_void_p(0x30000 + 512))
    assert rc == -3, msg


def test_forward_empty_is_ok(L):
    rc, msg = _fwd(L, B=0)
    assert rc == 0, msg
    rc, msg = _fwd(L, n=0, q=None, k=None, v=None, out=None)
    assert rc == 0, msg


def test_workspace_query(L):
    assert hla.forward_workspace_bytes(1, 16, 65536, 64, 64) > 0
    assert hla.forward_workspace_bytes(1, 1, 0, 64, 64) == 0
    with pytest.raises(ValueError):
        hla.forward_workspace_bytes(1, 1, 16, 40, 64)


@pytest.mark.parametrize("dtype, d, dv", [(torch.bfloat16, 128, 128), (torch.float32, 128, 128),
                                           (torch.float32, 64, 64)])
def test_wide_chunk_queries_agree_with_a_narrower_width(L, dtype, d, dv):
    """A chunk width whose tiles no kernel holds: the workspace and plan queries report the
    narrower width the call runs at (the same width for both), never an error."""
    plan128 = hla.forward_plan(2, 3, 1000, d, dv, 128, dtype, want_final_state=True)
    ws128 = hla.forward_workspace_bytes(2, 3, 1000, d, dv, 128, dtype, want_final_state=True)
    same = [W for W in (64, 32, 16)
            if hla.forward_plan(2, 3, 1000, d, dv, W, dtype, want_final_state=True) == plan128
            and hla.forward_workspace_bytes(2, 3, 1000, d, dv, W, dtype, want_final_state=True) == ws128]
    assert same and ws128 > 0


def test_decode_rejects_bad_arguments(L):
    o = Opts(1, 1e-6, None, 0, None, None)
    rc = L.hla2_decode_step(None, ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
                            ctypes.c_void_p(16), 1, 1, 16, 16, None, 0, None, ctypes.byref(o))
    assert rc == -1
    rc = L.hla2_decode_step(ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
                            ctypes.c_void_p(16), ctypes.c_void_p(16), 1, 1, 20, 16, None, 0, None,
                            ctypes.byref(o))
    assert rc == -1
    rc = L.hla2_decode_step(None, None, None, None, None, 0, 4, 16, 16, None, 0, None, ctypes.byref(o))
    assert rc == 0


def _bwd(L, **kw):
    # distinct (never dereferenced) addresses, 16-byte aligned
    names = ("q", "k", "v", "dout", "dq", "dk", "dv_out")
    args = {nm: ctypes.c_void_p(0x10000 * (i + 1)) for i, nm in enumerate(names)}
    args.update(B=1, H=2, n=16, d=16, dv=16, normalize=0, chunk=16, opts=Opts(1, 1e-6, None, 0, None, None))
    args.update(kw)
    o = args["opts"]
    rc = L.hla2_backward(*(args[nm] for nm in names), args["B"], args["H"], args["n"], args["d"], args["dv"],
                         None, args["normalize"], args["chunk"], None, None if o is None else ctypes.byref(o))
    return rc, L.hla2_last_error().decode()


def test_backward_empty_is_ok(L):
    """No heads or no tokens: nothing to compute, and the tensors may be NULL; the workspace
    query answers 0."""
    nulls = dict(q=None, k=None, v=None, dout=None, dq=None, dk=None, dv_out=None)
    for kw in (dict(B=0), dict(H=0), dict(n=0), dict(n=0, normalize=1)):
        rc, msg = _bwd(L, **kw, **nulls)
        assert rc == 0, (kw, msg)
    for normalize in (0, 1):
        assert L.hla2_backward_workspace_bytes(1, 2, 0, 64, 64, 64, 1, normalize) == 0
        assert L.hla2_backward_workspace_bytes(0, 2, 100, 64, 64, 64, 1, normalize) == 0


@pytest.mark.parametrize("kw", [
    dict(opts=None),
    dict(d=48),
    dict(chunk=24),
    dict(n=-1),
    dict(normalize=2),
    dict(dq=None),
    dict(dv_out=None),
    dict(dk=ctypes.c_void_p(0x10008)),                               # not 16-byte aligned
    dict(opts=Opts(1, 1e-6, None, 0, ctypes.c_void_p(16), None)),    # init_state
    dict(opts=Opts(1, 1e-6, None, 0, None, ctypes.c_void_p(16))),    # final_state
    dict(normalize=1, opts=Opts(1, float("nan"), None, 0, None, None)),
])
def test_backward_rejects_bad_arguments(L, kw):
    rc, msg = _bwd(L, **kw)
    assert rc == -1, msg
    assert msg


def test_normalized_backward_checks_before_launching(L):
    """The ratio-normalised backward is argument-checked on the host: it needs its larger
    workspace, finite eps, and cannot reuse saved (unnormalised) forward states."""
    p = ctypes.c_void_p(16)
    o = Opts(1, 1e-6, None, 0, None, None)
    rc = L.hla2_backward(p, p, p, p, p, p, p, 1, 1, 16, 16, 16, None, 1, 16, None, ctypes.byref(o))
    assert rc == -3 and b"workspace" in L.hla2_last_error()
    o = Opts(1, 1e-6, None, 0, None, None, None, 0, 2)
    rc = L.hla2_backward(p, p, p, p, p, p, p, 1, 1, 16, 16, 16, None, 1, 16, None, ctypes.byref(o))
    assert rc == -2
    n0 = L.hla2_backward_workspace_bytes(1, 2, 100, 32, 32, 32, 1, 0)
    n1 = L.hla2_backward_workspace_bytes(1, 2, 100, 32, 32, 32, 1, 1)
    assert 0 < n0 < n1 < 2**40
    # the bf16 tensor-core backward needs d == dv; float32 (SIMT) and the normalised
    # backward (which composes float32 passes) take any d, dv
    assert L.hla2_backward_workspace_bytes(1, 2, 100, 32, 16, 32, 1, 0) == ctypes.c_size_t(-1).value
    assert 0 < L.hla2_backward_workspace_bytes(1, 2, 100, 32, 16, 32, 1, 1) < 2**40
    assert 0 < L.hla2_backward_workspace_bytes(1, 2, 100, 32, 16, 32, 0, 0) < 2**40
    # float32 states: the fp32 backward's workspace is larger than the bf16 one's
    assert L.hla2_backward_workspace_bytes(1, 2, 100, 32, 32, 32, 0, 0) > n0


def test_unknown_flags_rejected(L):
    """Flag bits outside HLA2_FLAG_* are argument errors, found before anything runs."""
    p = ctypes.c_void_p(16)
    o = Opts(1, 1e-6, None, 0, None, None, None, 0, 4)
    rc = L.hla2_forward(p, p, p, p, 0, 1, 16, 16, 16, None, 0, 16, None, ctypes.byref(o))
    assert rc == -1 and b"flags" in L.hla2_last_error()
    o = Opts(1, 1e-6, None, 0, None, None, None, 0, 1)  # SAVE_FOR_BACKWARD is a forward flag
    rc = L.hla2_backward(p, p, p, p, p, p, p, 0, 1, 16, 16, 16, None, 0, 16, None, ctypes.byref(o))
    assert rc == -1
    o = Opts(1, 1e-6, None, 0, None, None, None, 0, 2)  # STATES_SAVED is a backward flag
    rc = L.hla2_forward(p, p, p, p, 0, 1, 16, 16, 16, None, 0, 16, None, ctypes.byref(o))
    assert rc == -1


def test_unmasked_flag_abi(L):
    """HLA2_FLAG_UNMASKED is accepted by the forward and the decode step, refused together
    with SAVE_FOR_BACKWARD (the backward covers the masked output), and bit 16 is unknown."""
    p = ctypes.c_void_p(16)
    o = Opts(1, 1e-6, None, 0, None, None, None, 0, 8)
    assert L.hla2_forward(p, p, p, p, 0, 1, 16, 16, 16, None, 0, 16, None, ctypes.byref(o)) == 0
    assert L.hla2_decode_step(p, p, p, p, p, 0, 1, 16, 16, None, 0, None, ctypes.byref(o)) == 0
    o = Opts(1, 1e-6, None, 0, None, None, None, 0, 8 | 4)
    assert L.hla2_decode_step(p, p, p, p, p, 0, 1, 16, 16, None, 0, None, ctypes.byref(o)) == 0
    o = Opts(1, 1e-6, None, 0, None, None, None, 0, 8 | 1)
    rc = L.hla2_forward(p, p, p, p, 1, 1, 16, 16, 16, None, 0, 16, None, ctypes.byref(o))
    assert rc == -2 and b"masked" in L.hla2_last_error()
    o = Opts(1, 1e-6, None, 0, None, None, None, 0, 16)
    assert L.hla2_forward(p, p, p, p, 0, 1, 16, 16, 16, None, 0, 16, None, ctypes.byref(o)) == -1
    assert L.hla2_decode_step(p, p, p, p, p, 0, 1, 16, 16, None, 0, None, ctypes.byref(o)) == -1


def test_multi_query_decode_abi(L):
    """hla2_decode_step_mq: group 1..8, no compact flag, head-state size C | G | m | h."""
    p = ctypes.c_void_p(16)
    assert L.hla2_mq_head_state_floats(128, 64) == 2 * 128 * 64 + 2 * 128
    o = Opts(1, 1e-6, None, 0, None, None, None, 0, 0)
    for group in (0, 9):
        rc = L.hla2_decode_step_mq(p, p, p, p, p, p, 1, 1, group, 16, 16, None, 0, None, ctypes.byref(o))
        assert rc == -1 and b"group" in L.hla2_last_error()
    assert L.hla2_decode_step_mq(p, p, p, p, p, p, 0, 4, 4, 16, 16, None, 0, None, ctypes.byref(o)) == 0
    o = Opts(1, 1e-6, None, 0, None, None, None, 0, 4)
    assert L.hla2_decode_step_mq(p, p, p, p, p, p, 1, 1, 2, 16, 16, None, 0, None, ctypes.byref(o)) == -2
    o = Opts(1, 1e-6, None, 0, None, None, None, 0, 8)
    assert L.hla2_decode_step_mq(p, p, p, p, p, p, 0, 1, 2, 16, 16, None, 0, None, ctypes.byref(o)) == 0
    rc = L.hla2_decode_step_mq(None, p, p, p, p, p, 1, 1, 2, 16, 16, None, 0, None, ctypes.byref(o))
    assert rc == -1


def test_compact_state_abi(L):
    from oracle import hla2_oracle as O

    for d, dv in ((16, 16), (64, 32), (128, 128)):
        assert L.hla2_compact_state_floats(d, dv) == O.compact_state_floats(d, dv)
    assert L.hla2_compact_state_floats(128, 128) == 41472  # 8448 for S instead of 16384
    p = ctypes.c_void_p(16)
    o = Opts(1, 1e-6, None, 0, None, None, None, 0, 1)  # a forward flag on the decode step
    rc = L.hla2_decode_step(p, p, p, p, p, 1, 1, 16, 16, None, 0, None, ctypes.byref(o))
    assert rc == -1 and b"flags" in L.hla2_last_error()
    assert L.hla2_state_to_compact(p, p, 1, 1, 20, 16, None) == -1      # bad d
    assert L.hla2_state_to_compact(None, None, 0, 4, 16, 16, None) == 0  # nothing to do
    assert L.hla2_state_from_compact(p, p, 1, 1, 16, 16, None) == -1     # overlapping buffers


def test_debug_queries_report_a_normal_build():
    """The normal build has no bounds checks: both debug entry points answer
    HLA2_ERR_UNSUPPORTED (without touching a device)."""
    L = hla.lib()
    assert L.hla2_debug_status(0) == -2
    assert b"debug build" in L.hla2_last_error()
    assert L.hla2_debug_selftest(None) == -2


def test_forward_plan_segments_cover_the_sequence():
    """Host-side segment plans (no device: the planner's GB300 defaults): for seeded random
    shapes the plan's segments of seg_chunks chunks, at some chunk width W <= chunk the kernels
    run at, cover the n tokens with no segment left empty; an empty sequence plans nothing."""
    import random

    rng = random.Random(0)
    checked = 0
    for _ in range(300):
        B, H, n = rng.randint(1, 4), rng.randint(1, 40), rng.randint(1, 70000)
        d = rng.choice([16, 32, 64, 128])
        dv = d if rng.random() < 0.7 else rng.choice([16, 32, 64, 128])
        chunk = rng.choice([16, 32, 64, 128])
        dtype = rng.choice([torch.bfloat16, torch.float32])
        normalize, final = rng.random() < 0.2, rng.random() < 0.3
        try:
            nseg, seg_chunks, launches = hla.forward_plan(B, H, n, d, dv, chunk, dtype, normalize, final)
        except (ValueError, hla.HLA2Error):
            continue  # shapes no kernel covers
        assert nseg >= 1 and seg_chunks >= 1 and launches >= 1
        assert any((nseg - 1) * seg_chunks * W < n <= nseg * seg_chunks * W for W in (16, 32, 64, 128) if W <= chunk), \
            (B, H, n, d, dv, chunk, dtype, normalize, final, nseg, seg_chunks)
        checked += 1
    assert checked > 200
    nseg, _, launches = hla.forward_plan(1, 1, 0, 64, 64, 128)
    assert nseg == 0 and launches == 0
