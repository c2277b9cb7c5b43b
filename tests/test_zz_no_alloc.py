"""The allocation-free forward entry point (hla2_forward_noalloc), through the C ABI.

It serves callers that cannot allocate device memory (hosts that pass a kernel only its
inputs and outputs, programs without a device allocator): its scratch is a fixed array inside
the library.  Its
output must match hla2_forward's (which takes a caller-provided workspace) and the float64
oracle's within the bf16 parity tolerance, on two calls in a row (the array keeps the
previous call's contents).  A bounded wait that gives up is reported through the array's
status word (hla2_noalloc_status).  This file is collected last so that a
stop-at-first-failure run has run everything else.
"""
import ctypes

import pytest
import torch

import chunked_scan_mixer_gb300 as hla
from chunked_scan_mixer_gb300 import inputs

from oracle import cref

from .helpers import np32, np64, rel_err

pytestmark = pytest.mark.gpu

HLA2_BF16 = 1
HLA2_ERR_WORKSPACE = -3
HLA2_ERR_TIMEOUT = -5


def noalloc(q, k, v, gamma, chunk, normalize=False):
    B, H, n, d = q.shape
    dv = v.shape[-1]
    out = torch.empty_like(v)
    rc = hla.lib().hla2_forward_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(out.data_ptr()), B, H, n, d, dv, ctypes.c_void_p(gamma.data_ptr()), int(normalize), chunk,
        HLA2_BF16, 1e-6, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, hla.lib().hla2_last_error().decode()
    return out


@pytest.mark.parametrize("chunk, normalize", [(128, False), (64, False), (64, True)])
def test_matches_workspace_entry_point_on_two_calls(chunk, normalize):
    x = inputs.make_custom(1, 4, 3000, 64, 64, torch.bfloat16, seed=31, gamma=(0.98, 0.9999),
                           qk="softplus" if normalize else "gauss")
    q, k, v, g = (x[n].cuda() for n in ("q", "k", "v", "gamma"))
    ref = np64(hla.forward(q, k, v, gamma=g, chunk=chunk, normalize=normalize).cpu())
    first = np64(noalloc(q, k, v, g, chunk, normalize).cpu())
    second = np64(noalloc(q, k, v, g, chunk, normalize).cpu())
    assert rel_err(first, ref) <= 2e-2
    assert rel_err(second, ref) <= 2e-2
    oracle = cref.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), x["gamma"].double().numpy(),
                          normalize=normalize, eps=1e-6)
    assert rel_err(first, oracle) <= 2e-2
    assert rel_err(second, oracle) <= 2e-2
    assert hla.lib().hla2_noalloc_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0


def test_timed_out_wait_in_its_scratch_is_reported():
    """The bounded-wait self-test run on the library's scratch array: the status query reports
    the timeout; the next call clears it and is correct again."""
    L = hla.lib()
    sh = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    x = inputs.make_custom(1, 2, 700, 64, 64, torch.bfloat16, seed=32, gamma=(0.97, 0.999))
    q, k, v, g = (x[n].cuda() for n in ("q", "k", "v", "gamma"))
    noalloc(q, k, v, g, 128)
    assert L.hla2_noalloc_status(sh) == 0
    assert L.hla2_noalloc_selftest_wait_timeout(sh) == 0
    assert L.hla2_noalloc_status(sh) == HLA2_ERR_TIMEOUT  # synchronises: the wait has given up
    assert b"site 90" in L.hla2_last_error()
    o = np64(noalloc(q, k, v, g, 128).cpu())
    assert L.hla2_noalloc_status(sh) == 0
    ref = cref.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), x["gamma"].double().numpy())
    assert rel_err(o, ref) <= 2e-2


def test_rejects_sizes_beyond_its_scratch():
    q = torch.empty(16, device="cuda", dtype=torch.bfloat16)  # never read: the size check comes first
    p = ctypes.c_void_p(q.data_ptr())
    rc = hla.lib().hla2_forward_noalloc(p, p, p, p, 4, 16, 8192, 128, 128, None, 0, 64, HLA2_BF16, 1e-6, None)
    assert rc == HLA2_ERR_WORKSPACE
    assert "scratch" in hla.lib().hla2_last_error().decode()
