"""Failure detection on the GPU without a fault: the bounded wait of the tcgen05 kernels is
made to run out on an mbarrier that nothing arrives at (hla2_selftest_wait_timeout); the
kernel records the site in the workspace status word and returns, the host reads
HLA2_ERR_TIMEOUT, and the context stays usable for the next call."""
import ctypes

import pytest
import torch

import chunked_scan_mixer_gb300 as hla
from chunked_scan_mixer_gb300 import inputs
from chunked_scan_mixer_gb300.hla2 import _stream_handle
from oracle import cref

from .helpers import np32, np64, rel_err

pytestmark = pytest.mark.gpu


def test_timed_out_wait_is_reported_and_the_context_survives():
    L = hla.lib()
    dev = torch.device("cuda", 0)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    sh = _stream_handle(dev)
    p = ctypes.c_void_p(ws.data_ptr())
    assert L.hla2_workspace_status(p, sh) == 0
    assert L.hla2_selftest_wait_timeout(p, sh) == 0
    rc = L.hla2_workspace_status(p, sh)  # synchronises: the wait has given up by now
    assert rc == -5, rc  # HLA2_ERR_TIMEOUT
    assert b"site 90" in L.hla2_last_error()
    # the context is still usable: a tcgen05 forward runs and matches the oracle
    x = inputs.make_custom(1, 2, 300, 64, 64, torch.bfloat16, seed=3, gamma=(0.97, 0.999))
    o = hla.forward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), gamma=x["gamma"].cuda(), chunk=128)
    hla.check_status()
    ref = cref.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), x["gamma"].double().numpy())
    assert rel_err(np64(o.cpu()), ref) <= 2e-2
