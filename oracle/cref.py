"""ctypes wrapper of the float64 C oracle (``hla2_oracle.c``).

TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the benchmark's
CPU legs.  ``build()`` compiles the C file with gcc and OpenMP into ``oracle/_build``.
The arithmetic is documented in the C file; this module only marshals arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hla2_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libhla2_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle (portable flags: the same source builds on x86-64 and Arm)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O3", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        L = ctypes.c_long
        I = ctypes.c_int
        D = ctypes.c_double
        lib.hla2_oracle_threads.restype = I
        lib.hla2_oracle_forward.argtypes = [P, P, P, P, L, L, L, I, I, P, I, D, P, P, I]
        lib.hla2_oracle_forward.restype = I
        lib.hla2_oracle_decode.argtypes = [P, P, P, P, P, L, L, I, I, P, I, D, I]
        lib.hla2_oracle_decode.restype = I
        lib.hla2_oracle_backward.argtypes = [P, P, P, P, P, P, P, L, L, L, I, I, P]
        lib.hla2_oracle_backward.restype = I
        _lib = lib
    return _lib


def _f32(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def threads() -> int:
    return int(_load().hla2_oracle_threads())


def forward(q, k, v, gamma=None, normalize=False, eps=1e-6, init_state=None,
            return_state=False, masked=True):
    """Serial float64 forward.  q, k [B,H,n,d]; v [B,H,n,dv]; init_state packed
    [B,H,d*d+2*d*dv+2*d] (decode layout) or None.  Returns out [B,H,n,dv] float64
    (and the packed final state when ``return_state``)."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, H, n, d = q.shape
    dv = v.shape[-1]
    sf = d * d + 2 * d * dv + 2 * d
    out = np.empty((B, H, n, dv), dtype=np.float64)
    g = None if gamma is None else _f64(gamma).reshape(H)
    init = None if init_state is None else _f64(init_state).reshape(B, H, sf)
    fin = np.empty((B, H, sf), dtype=np.float64) if return_state else None
    rc = _load().hla2_oracle_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B * H, H, n, d, dv,
                                     _ptr(g), int(bool(normalize)), float(eps), _ptr(init),
                                     _ptr(fin), int(bool(masked)))
    if rc != 0:
        raise RuntimeError(f"hla2_oracle_forward failed ({rc})")
    return (out, fin) if return_state else out


def decode_step(state, q, k, v, gamma=None, normalize=False, eps=1e-6, masked=True):
    """One serial step on packed states [N,H,sf] float64 (modified in place).
    q, k [N,H,d]; v [N,H,dv].  Returns out [N,H,dv] float64."""
    assert state.dtype == np.float64 and state.flags.c_contiguous
    q, k, v = _f32(q), _f32(k), _f32(v)
    N, H, d = q.shape
    dv = v.shape[-1]
    out = np.empty((N, H, dv), dtype=np.float64)
    g = None if gamma is None else _f64(gamma).reshape(H)
    rc = _load().hla2_oracle_decode(_ptr(state), _ptr(q), _ptr(k), _ptr(v), _ptr(out), N * H, H,
                                    d, dv, _ptr(g), int(bool(normalize)), float(eps),
                                    int(bool(masked)))
    if rc != 0:
        raise RuntimeError(f"hla2_oracle_decode failed ({rc})")
    return out


def backward_normalized(q, k, v, dout, gamma=None, eps=1e-6):
    """Ratio-normalised gradients from the C recurrence, by the quotient rule of
    ``hla2_oracle.serial_backward_normalized``: the unnormalised output num and the
    denominator den (the same recurrence with v -> 1) from the C forward, then the C
    reverse sweep once with (v, dO / (den + eps)) and once with
    (1, -(dO . num) / (den + eps)^2).  Returns (dq, dk, dv) float64."""
    q, k, v, dout = _f32(q), _f32(k), _f32(v), _f64(dout)
    ones = np.ones(v.shape[:-1] + (1,), dtype=np.float32)
    num = forward(q, k, v, gamma)
    den = forward(q, k, ones, gamma)[..., 0]
    inv = 1.0 / (den + eps)
    dnum = dout * inv[..., None]
    dden = -np.sum(dout * num, axis=-1) * inv * inv
    dq1, dk1, dv1 = backward(q, k, v, dnum, gamma)
    dq2, dk2, _ = backward(q, k, ones, dden[..., None], gamma)
    return dq1 + dq2, dk1 + dk2, dv1


def backward(q, k, v, dout, gamma=None):
    """Reverse sweep of the unnormalised serial recurrence: returns (dq, dk, dv) float64."""
    q, k, v, dout = _f32(q), _f32(k), _f32(v), _f32(dout)
    B, H, n, d = q.shape
    dv = v.shape[-1]
    dq = np.empty((B, H, n, d), dtype=np.float64)
    dk = np.empty((B, H, n, d), dtype=np.float64)
    dvv = np.empty((B, H, n, dv), dtype=np.float64)
    g = None if gamma is None else _f64(gamma).reshape(H)
    rc = _load().hla2_oracle_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk),
                                      _ptr(dvv), B * H, H, n, d, dv, _ptr(g))
    if rc != 0:
        raise RuntimeError(f"hla2_oracle_backward failed ({rc})")
    return dq, dk, dvv
