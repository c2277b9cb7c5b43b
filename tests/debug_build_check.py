"""Runs the small odd shapes on the bounds-checking build (HLA2_DEBUG) of the library, in its
own process: every call is compared with the float64 oracle at the parity bar, and the debug
words must stay clean (no global-memory index outside its buffer).  Then the check's own
recording is exercised with hla2_debug_selftest (a failing check that guards no access).

    python tests/debug_build_check.py <path of the debug libhla2.so>

Prints DEBUG_BUILD_OK and exits 0 on success.  Used by tests/test_debug_build_gpu.py.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import chunked_scan_mixer_gb300.hla2 as H  # noqa: E402

H.LIB_PATH = sys.argv[1]
import chunked_scan_mixer_gb300 as hla  # noqa: E402
from chunked_scan_mixer_gb300 import inputs  # noqa: E402
from oracle import cref  # noqa: E402


def rel(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


def f32(t):
    return t.detach().to("cpu", torch.float32).numpy()


def tol(dtype):
    return 1e-4 if dtype == torch.float32 else 2e-2


def main():
    L = hla.lib()
    assert L.hla2_debug_status(1) == 0, "debug words not clean at start"
    cases = 0
    # forward: d = 16 with n = w and ragged tails, every chunk width, both dtypes, normalised too
    for dtype in (torch.float32, torch.bfloat16):
        for d, dv, chunk, n in ((16, 16, 16, 16), (16, 16, 16, 37), (16, 32, 32, 70), (32, 16, 64, 129),
                                (64, 64, 64, 200), (128, 128, 64, 131)):
            for normalize in (False, True):
                x = inputs.make_custom(1, 3, n, d, dv, dtype, seed=n + d, gamma=(0.9, 0.999),
                                       qk="softplus" if normalize else "gauss")
                o, fin = hla.forward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), gamma=x["gamma"].cuda(),
                                     chunk=chunk, normalize=normalize, return_final_state=True)
                ref, ref_state = cref.forward(f32(x["q"]), f32(x["k"]), f32(x["v"]), x["gamma"].double().numpy(),
                                              normalize=normalize, return_state=True)
                e = rel(f32(o), ref)
                assert e <= tol(dtype), ("forward", dtype, d, dv, chunk, n, normalize, e)
                cases += 1
    # backward: bf16 (mma.sync, and tcgen05 first-order scans at d = 128, chunk 128), float32 (SIMT)
    for dtype, d, chunk, n in ((torch.bfloat16, 16, 16, 16), (torch.bfloat16, 16, 16, 45), (torch.bfloat16, 64, 64, 150),
                               (torch.float32, 16, 16, 37), (torch.float32, 32, 32, 100),
                               (torch.bfloat16, 128, 128, 300)):
        x = inputs.make_custom(1, 2, n, d, d, dtype, seed=3 * n + d, gamma=(0.95, 0.999), with_dout=True)
        got = hla.backward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["dout"].cuda(), gamma=x["gamma"].cuda(),
                           chunk=chunk)
        refs = cref.backward(f32(x["q"]), f32(x["k"]), f32(x["v"]), f32(x["dout"]), x["gamma"].double().numpy())
        for name, gg, rr in zip(("dq", "dk", "dv"), got, refs):
            e = rel(f32(gg), rr)
            assert e <= tol(dtype), ("backward", name, dtype, d, chunk, n, e)
        cases += 1
    # decode: packed and compact state at d = 16, multi-query at d = 16
    N, Hh, d = 2, 4, 16
    x = inputs.make_custom(N, Hh, 20, d, d, torch.float32, seed=7, gamma=0.97)
    _, st = cref.forward(f32(x["q"]), f32(x["k"]), f32(x["v"]), x["gamma"].double().numpy(), return_state=True)
    packed = torch.from_numpy(st.astype(np.float32)).cuda()
    compact = hla.state_to_compact(packed, d, d)
    st_ref = st.astype(np.float32).astype(np.float64).copy()
    for step in range(3):
        q, k, v = inputs.decode_step_inputs(step, N, Hh, d, d, dtype=torch.float32)
        o1 = hla.decode_step(packed, q.cuda(), k.cuda(), v.cuda(), gamma=x["gamma"].cuda())
        o2 = hla.decode_step(compact, q.cuda(), k.cuda(), v.cuda(), gamma=x["gamma"].cuda(), compact=True)
        ref = cref.decode_step(st_ref, f32(q), f32(k), f32(v), x["gamma"].double().numpy())
        assert rel(f32(o1), ref) <= 1e-4 and rel(f32(o2), ref) <= 1e-4, ("decode", step)
        cases += 1
    key_state, head_state = hla.mq_split_state(torch.zeros((N, Hh, hla.state_floats(d, d)), device="cuda"), d, d, 2)
    q, _, _ = inputs.decode_step_inputs(9, N, Hh, d, d, dtype=torch.float32)
    _, k, v = inputs.decode_step_inputs(19, N, Hh // 2, d, d, dtype=torch.float32)
    o = hla.decode_step_mq(key_state, head_state, q.cuda(), k.cuda(), v.cuda(), gamma=0.99)
    ref = cref.decode_step(np.zeros((N, Hh, hla.state_floats(d, d))), f32(q), f32(k.repeat_interleave(2, dim=1)),
                           f32(v.repeat_interleave(2, dim=1)), np.full(Hh, 0.99))
    assert rel(f32(o), ref) <= 1e-4, "multi-query decode"
    cases += 1
    site = L.hla2_debug_status(1)
    assert site == 0, f"a bounds check failed at site {site}"
    # the recording itself: one failing check that guards no access
    assert L.hla2_debug_selftest(None) == 0
    assert L.hla2_debug_status(1) == 1
    assert L.hla2_debug_status(0) == 0  # cleared
    print(f"DEBUG_BUILD_OK {cases} cases")


if __name__ == "__main__":
    main()
