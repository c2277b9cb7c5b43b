"""Python binding of the HLA-2 C ABI (include/hla2.h).

Argument marshalling only: every step of the computation runs in the CUDA library
``_build/libhla2.so``.  PyTorch provides device memory and streams.  If the library
has not been built, every call raises ``RuntimeError``; there is no other code path.

Tensors given on the CPU are copied to the current CUDA device, processed there and
copied back (the end-to-end path); CUDA tensors are processed in place on the
current stream.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libhla2.so")

HLA2_F32 = 0
HLA2_BF16 = 1
_DTYPES = {torch.float32: HLA2_F32, torch.bfloat16: HLA2_BF16}

_lib = None
_lib_lock = threading.Lock()


class HLA2Error(RuntimeError):
    """A C-ABI call returned an error code."""

    def __init__(self, func, code, message):
        super().__init__(f"{func} failed with code {code}: {message}")
        self.code = code


class Opts(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int),
        ("eps", ctypes.c_float),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("init_state", ctypes.c_void_p),
        ("final_state", ctypes.c_void_p),
        ("phase_events", ctypes.POINTER(ctypes.c_void_p)),
        ("n_phase_events", ctypes.c_int),
        ("flags", ctypes.c_int),
    ]


FLAG_SAVE_FOR_BACKWARD = 1
FLAG_STATES_SAVED = 2


class SavedForBackward:
    """What a training-step forward keeps for the backward on the same inputs: a device
    workspace holding the segment summaries and the bf16 (S, Z) at every chunk start.
    Pass it to backward(saved=...) once; the buffer is owned by this object."""

    def __init__(self, ws, nbytes, key):
        self.ws, self.nbytes, self.key = ws, nbytes, key


def lib():
    """Load libhla2.so (once).  Raises RuntimeError when it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    with _lib_lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"HLA-2 CUDA library not found at {LIB_PATH}; build it with "
                "`python -m chunked_scan_mixer_gb300.build` (there is no fallback)")
        L = ctypes.CDLL(LIB_PATH)
        P, I, Z, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
        L.hla2_version.restype = I
        L.hla2_last_error.restype = ctypes.c_char_p
        L.hla2_state_floats.argtypes = [I, I]
        L.hla2_state_floats.restype = Z
        L.hla2_forward_workspace_bytes.argtypes = [I, I, I, I, I, I, I, I, I]
        L.hla2_forward_workspace_bytes.restype = Z
        L.hla2_forward.argtypes = [P, P, P, P, I, I, I, I, I, P, I, I, P, ctypes.POINTER(Opts)]
        L.hla2_forward.restype = I
        L.hla2_forward_plan.argtypes = [I, I, I, I, I, I, I, I, I, ctypes.POINTER(I), ctypes.POINTER(I),
                                        ctypes.POINTER(I)]
        L.hla2_forward_plan.restype = I
        L.hla2_workspace_status.argtypes = [P, P]
        L.hla2_workspace_status.restype = I
        L.hla2_backward_workspace_bytes.argtypes = [I, I, I, I, I, I, I, I]
        L.hla2_backward_workspace_bytes.restype = Z
        L.hla2_backward.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, P, I, I, P, ctypes.POINTER(Opts)]
        L.hla2_backward.restype = I
        L.hla2_decode_step.argtypes = [P, P, P, P, P, I, I, I, I, P, I, P, ctypes.POINTER(Opts)]
        L.hla2_decode_step.restype = I
        L.hla2_forward_noalloc.argtypes = [P, P, P, P, I, I, I, I, I, P, I, I, I, F, P]
        L.hla2_forward_noalloc.restype = I
        L.hla2_noalloc_status.argtypes = [P]
        L.hla2_noalloc_status.restype = I
        L.hla2_noalloc_selftest_wait_timeout.argtypes = [P]
        L.hla2_noalloc_selftest_wait_timeout.restype = I
        L.hla2_debug_status.argtypes = [I]
        L.hla2_debug_status.restype = I
        L.hla2_debug_selftest.argtypes = [P]
        L.hla2_debug_selftest.restype = I
        L.hla2_ahla_forward_workspace_bytes.argtypes = [I, I, I, I, I, I, I, I]
        L.hla2_ahla_forward_workspace_bytes.restype = Z
        L.hla2_ahla_forward.argtypes = [P, P, P, P, I, I, I, I, I, P, I, I, P, ctypes.POINTER(Opts)]
        L.hla2_ahla_forward.restype = I
        L.hla2_ahla_state_floats.argtypes = [I, I]
        L.hla2_ahla_state_floats.restype = Z
        L.hla2_ahla_decode_step.argtypes = [P, P, P, P, P, I, I, I, I, P, I, P, ctypes.POINTER(Opts)]
        L.hla2_ahla_decode_step.restype = I
        L.hla2_compact_state_floats.argtypes = [I, I]
        L.hla2_compact_state_floats.restype = Z
        L.hla2_hla3_forward_workspace_bytes.argtypes = [I, I, I, I, I, I, I, I, I]
        L.hla2_hla3_forward_workspace_bytes.restype = Z
        L.hla2_hla3_forward.argtypes = [P, P, P, P, I, I, I, I, I, P, I, I, P, ctypes.POINTER(Opts)]
        L.hla2_hla3_forward.restype = I
        L.hla2_ahla_backward_workspace_bytes.argtypes = [I, I, I, I, I, I, I, I]
        L.hla2_ahla_backward_workspace_bytes.restype = Z
        L.hla2_ahla_backward.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, P, I, I, P, ctypes.POINTER(Opts)]
        L.hla2_ahla_backward.restype = I
        L.hla2_hla3_decode_step.argtypes = [P, P, P, P, P, I, I, I, I, I, P, ctypes.POINTER(Opts)]
        L.hla2_hla3_decode_step.restype = I
        L.hla2_selftest_wait_timeout.argtypes = [P, P]
        L.hla2_selftest_wait_timeout.restype = I
        L.hla2_mq_head_state_floats.argtypes = [I, I]
        L.hla2_mq_head_state_floats.restype = Z
        L.hla2_decode_step_mq.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, I, P, ctypes.POINTER(Opts)]
        L.hla2_decode_step_mq.restype = I
        for name in ("hla2_state_to_compact", "hla2_state_from_compact"):
            getattr(L, name).argtypes = [P, P, I, I, I, I, P]
            getattr(L, name).restype = I
        _lib = L
        return L


EXPORTED_SYMBOLS = (
    "hla2_version", "hla2_last_error", "hla2_state_floats", "hla2_forward_workspace_bytes",
    "hla2_forward", "hla2_forward_plan", "hla2_workspace_status", "hla2_backward_workspace_bytes",
    "hla2_backward", "hla2_decode_step", "hla2_forward_noalloc", "hla2_compact_state_floats",
    "hla2_state_to_compact", "hla2_state_from_compact", "hla2_ahla_forward_workspace_bytes", "hla2_ahla_forward",
    "hla2_ahla_state_floats", "hla2_ahla_decode_step", "hla2_mq_head_state_floats", "hla2_decode_step_mq",
    "hla2_selftest_wait_timeout", "hla2_hla3_forward_workspace_bytes", "hla2_hla3_forward", "hla2_hla3_decode_step",
    "hla2_ahla_backward_workspace_bytes", "hla2_ahla_backward", "hla2_noalloc_status",
    "hla2_noalloc_selftest_wait_timeout", "hla2_debug_status", "hla2_debug_selftest",
)

FLAG_COMPACT_STATE = 4
FLAG_UNMASKED = 8


def _check(func, rc):
    if rc != 0:
        raise HLA2Error(func, rc, lib().hla2_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


_ws_cache: dict = {}


def _workspace(nbytes, device, stream_handle):
    """Scratch reused per (device, stream); grown on demand."""
    if nbytes == 0:
        return None
    key = (device.index, stream_handle.value)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


def check_status(device=None):
    """Raise HLA2Error if a kernel that used this stream's cached workspace reported a
    timed-out wait.  Synchronises the current stream."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    sh = _stream_handle(device)
    buf = _ws_cache.get((device.index, sh.value))
    if buf is not None:
        _check("hla2_workspace_status", lib().hla2_workspace_status(ctypes.c_void_p(buf.data_ptr()), sh))


def state_floats(d, dv, compact=False):
    """Floats in one head's decode state (packed layout, or the compact one)."""
    return int(lib().hla2_compact_state_floats(d, dv) if compact else lib().hla2_state_floats(d, dv))


def _convert_state(src, d, dv, to_compact):
    if src.device.type != "cuda" or src.dtype != torch.float32 or not src.is_contiguous():
        raise ValueError("state must be a contiguous float32 CUDA tensor")
    N, H = src.shape[:2]
    dst = torch.empty((N, H, state_floats(d, dv, compact=to_compact)), dtype=torch.float32, device=src.device)
    fn = lib().hla2_state_to_compact if to_compact else lib().hla2_state_from_compact
    _check(fn.__name__, fn(_ptr(src), _ptr(dst), N, H, d, dv, _stream_handle(src.device)))
    return dst


def state_to_compact(state, d, dv):
    """[N, H, state_floats(d, dv)] packed states -> [N, H, state_floats(d, dv, compact=True)]."""
    return _convert_state(state, d, dv, True)


def state_from_compact(compact, d, dv):
    """Compact states -> packed states (S mirrored from its stored upper block triangle)."""
    return _convert_state(compact, d, dv, False)


def forward_workspace_bytes(B, H, n, d, dv, chunk=64, dtype=torch.bfloat16, normalize=False,
                            want_final_state=False):
    r = lib().hla2_forward_workspace_bytes(B, H, n, d, dv, chunk, _DTYPES[dtype], int(normalize),
                                           int(want_final_state))
    if r == ctypes.c_size_t(-1).value:
        raise ValueError("arguments rejected by hla2_forward")
    return int(r)


def forward_plan(B, H, n, d, dv, chunk=64, dtype=torch.bfloat16, normalize=False, want_final_state=False):
    """(segments per head, chunks per segment, kernel launches per call)."""
    ns, sc, nl = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check("hla2_forward_plan", lib().hla2_forward_plan(B, H, n, d, dv, chunk, _DTYPES[dtype], int(normalize),
                                                        int(want_final_state), ctypes.byref(ns),
                                                        ctypes.byref(sc), ctypes.byref(nl)))
    return ns.value, sc.value, nl.value


def _gamma_tensor(gamma, H, device):
    if gamma is None:
        return None
    g = torch.as_tensor(gamma, dtype=torch.float32)
    if g.numel() == 1 and H != 1:
        g = g.reshape(1).expand(H)
    g = g.reshape(H).to(device=device, dtype=torch.float32).contiguous()
    return g


def _to_device(t, device):
    if t is None:
        return None
    if t.device.type == "cuda":
        return t.contiguous()
    return t.contiguous().to(device, non_blocking=True)


_side_streams: dict = {}
HOST_GROUPS = 8  # head groups of the pipelined host-tensor forward


def _pipelined_host_forward(q, k, v, gamma, normalize, chunk, eps, out, masked=True):
    """forward() on host tensors, overlapping the copies with the computation: the heads are
    independent, so they go through in groups -- the inputs of group i+1 are copied in on one
    stream while group i is computed on the current stream and group i-1's output is copied
    out on a third (two device buffers per group slot).  Returns None when the heads cannot
    be cut into at least two groups."""
    B, H, n, d = q.shape
    dv = v.shape[-1]
    # heads per group: a divisor of H giving at least HOST_GROUPS groups (the copies then
    # bound the call to within a group's compute and output copy of the link time), at
    # least two
    divisors = [c for c in range(H, 0, -1) if H % c == 0]
    gh = next((c for c in divisors if B * H // c >= HOST_GROUPS), next((c for c in divisors if B * H // c >= 2), 0))
    if gh == 0 or not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        return None
    device = torch.device("cuda", torch.cuda.current_device())
    key = device.index
    if key not in _side_streams:
        _side_streams[key] = (torch.cuda.Stream(device=device), torch.cuda.Stream(device=device))
    s_in, s_out = _side_streams[key]
    cur = torch.cuda.current_stream(device)
    g = _gamma_tensor(gamma, H, device)
    res = out if out is not None else torch.empty((B, H, n, dv), dtype=q.dtype, pin_memory=True)
    qf, kf, vf, rf = (t.view(B * H, n, t.shape[-1]) for t in (q, k, v, res))
    stage = [[torch.empty((gh, n, x), dtype=q.dtype, device=device) for x in (d, d, dv, dv)] for _ in range(2)]
    ev_in, ev_comp, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))
    s_in.wait_stream(cur)
    s_out.wait_stream(cur)
    for i, r0 in enumerate(range(0, B * H, gh)):
        slot, r1, h0 = i % 2, r0 + gh, r0 % H
        qd, kd, vd, od = stage[slot]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_comp[slot])  # group i-2 has read its inputs
            qd.copy_(qf[r0:r1], non_blocking=True)
            kd.copy_(kf[r0:r1], non_blocking=True)
            vd.copy_(vf[r0:r1], non_blocking=True)
            ev_in[slot].record(s_in)
        cur.wait_event(ev_in[slot])
        if i >= 2:
            cur.wait_event(ev_out[slot])  # group i-2's output has left this slot
        forward(qd.view(1, gh, n, d), kd.view(1, gh, n, d), vd.view(1, gh, n, dv),
                gamma=None if g is None else g[h0:h0 + gh], normalize=normalize, chunk=chunk, eps=eps,
                out=od.view(1, gh, n, dv), masked=masked)
        ev_comp[slot].record(cur)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[slot])
            rf[r0:r1].copy_(od, non_blocking=True)
            ev_out[slot].record(s_out)
    cur.wait_stream(s_in)
    cur.wait_stream(s_out)
    cur.synchronize()
    return res


def forward(q, k, v, gamma=None, normalize=False, chunk=64, eps=1e-6, init_state=None,
            return_final_state=False, out=None, phase_events=None, save_for_backward=False, masked=True):
    """Masked HLA-2 forward.  q, k [B,H,n,d]; v [B,H,n,dv] (float32 or bfloat16).
    masked=False computes the unmasked output q^T S C instead (HLA2_FLAG_UNMASKED).

    gamma: None, a scalar, or [H] per-head decay in (0, 1].  init_state: packed
    [B,H,state_floats] float32 state to continue from.  Returns out [B,H,n,dv] (and the
    packed final state when ``return_final_state``).  phase_events: optional list of
    torch.cuda.Event recorded at the phase boundaries (see hla2_opts).
    save_for_backward: also return a SavedForBackward for backward(saved=...), which then
    skips recomputing the forward (bf16 device tensors, unnormalised, no state arguments)."""
    host = q.device.type == "cpu"
    device = torch.device("cuda", torch.cuda.current_device()) if host else q.device
    L = lib()
    if q.dtype not in _DTYPES or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must all be float32 or all bfloat16")
    if (host and init_state is None and not return_final_state and phase_events is None and not save_for_backward
            and k.device.type == "cpu" and v.device.type == "cpu" and (out is None or out.device.type == "cpu")):
        res = _pipelined_host_forward(q, k, v, gamma, normalize, chunk, eps, out, masked)
        if res is not None:
            return res
    B, H, n, d = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != q.shape[:3]:
        raise ValueError("shape mismatch between q, k, v")
    qd, kd, vd = (_to_device(t, device) for t in (q, k, v))
    g = _gamma_tensor(gamma, H, device)
    init = None
    if init_state is not None:
        init = _to_device(init_state, device).to(torch.float32).contiguous()
        if init.shape != (B, H, state_floats(d, dv)):
            raise ValueError("init_state must be [B, H, state_floats(d, dv)]")
    o = out if (out is not None and not host) else torch.empty((B, H, n, dv), dtype=q.dtype, device=device)
    fin = torch.empty((B, H, state_floats(d, dv)), dtype=torch.float32, device=device) \
        if return_final_state else None
    sh = _stream_handle(device)
    flags = 0 if masked else FLAG_UNMASKED
    if save_for_backward:
        if host:
            raise ValueError("save_for_backward needs device tensors")
        nbytes = L.hla2_backward_workspace_bytes(B, H, n, d, dv, chunk, _DTYPES[q.dtype], 0)
        if nbytes == ctypes.c_size_t(-1).value:
            raise HLA2Error("hla2_backward_workspace_bytes", -2, "these arguments have no backward")
        ws = torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)
        flags |= FLAG_SAVE_FOR_BACKWARD
    else:
        nbytes = forward_workspace_bytes(B, H, n, d, dv, chunk, q.dtype, normalize, return_final_state)
        ws = _workspace(nbytes, device, sh)
    opts = Opts(_DTYPES[q.dtype], float(eps), None if ws is None else ws.data_ptr(), nbytes,
                None if init is None else init.data_ptr(), None if fin is None else fin.data_ptr(),
                None, 0, flags)
    if phase_events:
        for e in phase_events:
            if not e.cuda_event:  # torch creates its events lazily
                e.record()
        ev = (ctypes.c_void_p * len(phase_events))(*[e.cuda_event for e in phase_events])
        opts.phase_events = ctypes.cast(ev, ctypes.POINTER(ctypes.c_void_p))
        opts.n_phase_events = len(phase_events)
    rc = L.hla2_forward(_ptr(qd), _ptr(kd), _ptr(vd), _ptr(o), B, H, n, d, dv, _ptr(g), int(normalize),
                        chunk, sh, ctypes.byref(opts))
    _check("hla2_forward", rc)
    if save_for_backward:
        saved = SavedForBackward(ws, int(nbytes), (B, H, n, d, dv, chunk, q.dtype, device))
        return (o, fin, saved) if return_final_state else (o, saved)
    if host:
        o = o.to("cpu") if out is None else out.copy_(o)
        fin = None if fin is None else fin.to("cpu")
    return (o, fin) if return_final_state else o


def ahla_state_floats(d, dv):
    return int(lib().hla2_ahla_state_floats(d, dv))


def ahla_forward(q, k, v, gamma=None, normalize=False, chunk=64, eps=1e-6, out=None, phase_events=None,
                 return_final_state=False, init_state=None):
    """Asymmetric HLA forward (the masked left-cascaded product Q (K^T Q)(K^T V)).
    bf16 q, k, v [B,H,n,d] on the GPU (d == dv); chunk 32 or 64 (or 128 at d = 64,
    unnormalised).  Returns out [B,H,n,d] (and, with return_final_state, the state
    [B,H,ahla_state_floats] = P | E | m | n after the last token; a chunk-128 call with a final
    state runs at width 64).
    init_state: a state in that layout to continue from."""
    L = lib()
    if q.device.type != "cuda" or q.dtype != torch.bfloat16 or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must be bfloat16 CUDA tensors")
    B, H, n, d = q.shape
    dv = v.shape[-1]
    device = q.device
    qd, kd, vd = (t.contiguous() for t in (q, k, v))
    g = _gamma_tensor(gamma, H, device)
    o = out if out is not None else torch.empty((B, H, n, dv), dtype=q.dtype, device=device)
    sh = _stream_handle(device)
    nbytes = L.hla2_ahla_forward_workspace_bytes(B, H, n, d, dv, chunk, _DTYPES[q.dtype], int(normalize))
    if nbytes == ctypes.c_size_t(-1).value:
        nbytes = 0
    ws = _workspace(int(nbytes), device, sh)
    fin = torch.empty((B, H, ahla_state_floats(d, dv)), dtype=torch.float32, device=device) \
        if return_final_state else None
    init = None
    if init_state is not None:
        init = init_state.to(device=device, dtype=torch.float32).contiguous()
        if init.shape != (B, H, ahla_state_floats(d, dv)):
            raise ValueError("init_state must be [B, H, ahla_state_floats(d, dv)]")
    opts = Opts(_DTYPES[q.dtype], float(eps), None if ws is None else ws.data_ptr(), int(nbytes),
                None if init is None else init.data_ptr(), None if fin is None else fin.data_ptr(), None, 0, 0)
    if phase_events:
        for e in phase_events:
            if not e.cuda_event:
                e.record()
        ev = (ctypes.c_void_p * len(phase_events))(*[e.cuda_event for e in phase_events])
        opts.phase_events = ctypes.cast(ev, ctypes.POINTER(ctypes.c_void_p))
        opts.n_phase_events = len(phase_events)
    _check("hla2_ahla_forward", L.hla2_ahla_forward(_ptr(qd), _ptr(kd), _ptr(vd), _ptr(o), B, H, n, d, dv, _ptr(g),
                                                    int(normalize), chunk, sh, ctypes.byref(opts)))
    return (o, fin) if return_final_state else o


def ahla_decode_step(state, q, k, v, gamma=None, normalize=False, eps=1e-6, out=None):
    """One AHLA step; ``state`` [N,H,ahla_state_floats] float32 on the GPU is updated in
    place.  q, k [N,H,d]; v [N,H,dv].  Returns out [N,H,dv]."""
    L = lib()
    if state.device.type != "cuda" or state.dtype != torch.float32 or not state.is_contiguous():
        raise ValueError("state must be a contiguous float32 CUDA tensor")
    device = state.device
    N, H, d = q.shape
    dv = v.shape[-1]
    qd, kd, vd = (_to_device(t, device) for t in (q, k, v))
    g = _gamma_tensor(gamma, H, device)
    o = out if out is not None else torch.empty((N, H, dv), dtype=q.dtype, device=device)
    opts = Opts(_DTYPES[q.dtype], float(eps), None, 0, None, None, None, 0, 0)
    _check("hla2_ahla_decode_step", L.hla2_ahla_decode_step(_ptr(state), _ptr(qd), _ptr(kd), _ptr(vd), _ptr(o), N, H,
                                                            d, dv, _ptr(g), int(normalize), _stream_handle(device),
                                                            ctypes.byref(opts)))
    return o


def backward(q, k, v, dout, gamma=None, chunk=64, dq=None, dk=None, dv=None, saved=None, normalize=False,
             eps=1e-6):
    """Gradients (dq, dk, dv) for upstream dout of the unnormalised forward, or with
    ``normalize`` of the ratio-normalised one (o / (den + eps)).  saved: the
    SavedForBackward of forward(..., save_for_backward=True) on the same q, k, v, gamma
    and chunk (the forward is then not recomputed; unnormalised only)."""
    host = q.device.type == "cpu"
    device = torch.device("cuda", torch.cuda.current_device()) if host else q.device
    L = lib()
    B, H, n, d = q.shape
    dvdim = v.shape[-1]
    qd, kd, vd, dod = (_to_device(t, device) for t in (q, k, v, dout))
    g = _gamma_tensor(gamma, H, device)
    gq = torch.empty_like(qd) if dq is None or host else dq
    gk = torch.empty_like(kd) if dk is None or host else dk
    gv = torch.empty_like(vd) if dv is None or host else dv
    sh = _stream_handle(device)
    flags = 0
    if saved is not None:
        if saved.key != (B, H, n, d, dvdim, chunk, q.dtype, device):
            raise ValueError("saved was made for other sizes, chunk, dtype or device")
        ws, nbytes, flags = saved.ws, saved.nbytes, FLAG_STATES_SAVED
    else:
        nbytes = L.hla2_backward_workspace_bytes(B, H, n, d, dvdim, chunk, _DTYPES[q.dtype], int(normalize))
        if nbytes == ctypes.c_size_t(-1).value:
            nbytes = 0
        ws = _workspace(int(nbytes), device, sh)
    opts = Opts(_DTYPES[q.dtype], float(eps), None if ws is None else ws.data_ptr(), int(nbytes), None, None,
                None, 0, flags)
    rc = L.hla2_backward(_ptr(qd), _ptr(kd), _ptr(vd), _ptr(dod), _ptr(gq), _ptr(gk), _ptr(gv), B, H, n, d,
                         dvdim, _ptr(g), int(normalize), chunk, sh, ctypes.byref(opts))
    _check("hla2_backward", rc)
    if host:
        return gq.cpu(), gk.cpu(), gv.cpu()
    return gq, gk, gv


def decode_step(state, q, k, v, gamma=None, normalize=False, eps=1e-6, out=None, compact=False, masked=True):
    """One decode step; ``state`` [N,H,state_floats(d, dv, compact)] float32 on the GPU is
    updated in place (compact: the block-triangular S layout).  q, k [N,H,d]; v [N,H,dv].
    masked=False: the unmasked output q^T S C (G and h untouched).  Returns out [N,H,dv]."""
    L = lib()
    if state.device.type != "cuda" or state.dtype != torch.float32 or not state.is_contiguous():
        raise ValueError("state must be a contiguous float32 CUDA tensor")
    device = state.device
    N, H, d = q.shape
    dv = v.shape[-1]
    qd, kd, vd = (_to_device(t, device) for t in (q, k, v))
    g = _gamma_tensor(gamma, H, device)
    o = out if out is not None else torch.empty((N, H, dv), dtype=q.dtype, device=device)
    flags = (FLAG_COMPACT_STATE if compact else 0) | (0 if masked else FLAG_UNMASKED)
    opts = Opts(_DTYPES[q.dtype], float(eps), None, 0, None, None, None, 0, flags)
    rc = L.hla2_decode_step(_ptr(state), _ptr(qd), _ptr(kd), _ptr(vd), _ptr(o), N, H, d, dv, _ptr(g),
                            int(normalize), _stream_handle(device), ctypes.byref(opts))
    _check("hla2_decode_step", rc)
    return o


def mq_head_state_floats(d, dv):
    """Floats of one head's part of the multi-query state: C | G | m | h."""
    return int(lib().hla2_mq_head_state_floats(d, dv))


def mq_split_state(state, d, dv, group):
    """Packed per-head states [N, H, state_floats(d, dv)] whose heads share S within groups of
    ``group`` (e.g. a forward's final state on keys repeated over each group's heads) ->
    (key_state [N, H/group, d*d], head_state [N, H, mq_head_state_floats(d, dv)]).  S is
    taken from each group's first head; a layout copy only (the packed order is
    S | C | G | m | h, so a head's part is the tail after S)."""
    N, H, sf = state.shape
    if sf != state_floats(d, dv) or H % group:
        raise ValueError("state must be [N, H, state_floats(d, dv)] with H a multiple of group")
    return state[:, ::group, :d * d].contiguous(), state[:, :, d * d:].contiguous()


def mq_merge_state(key_state, head_state, d, dv):
    """Inverse of mq_split_state: packed per-head states with each group's S repeated."""
    N, Hk, _ = key_state.shape
    H = head_state.shape[1]
    S = key_state.repeat_interleave(H // Hk, dim=1)
    return torch.cat([S, head_state], dim=-1).contiguous()


def decode_step_mq(key_state, head_state, q, k, v, gamma=None, normalize=False, eps=1e-6, out=None, masked=True):
    """One decode step with one key moment per key group (multi-query sharing).
    key_state [N,Hk,d*d] and head_state [N,H,mq_head_state_floats(d, dv)] float32 on the GPU
    are updated in place; q [N,H,d] with H = Hk * group; k [N,Hk,d]; v [N,Hk,dv];
    gamma None, a scalar or [Hk].  Returns out [N,H,dv]."""
    L = lib()
    for t in (key_state, head_state):
        if t.device.type != "cuda" or t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError("states must be contiguous float32 CUDA tensors")
    device = key_state.device
    N, H, d = q.shape
    Hk, dv = k.shape[1], v.shape[-1]
    if H % Hk:
        raise ValueError("the query heads must be a multiple of the key heads")
    group = H // Hk
    qd, kd, vd = (_to_device(t, device) for t in (q, k, v))
    g = _gamma_tensor(gamma, Hk, device)
    o = out if out is not None else torch.empty((N, H, dv), dtype=q.dtype, device=device)
    opts = Opts(_DTYPES[q.dtype], float(eps), None, 0, None, None, None, 0, 0 if masked else FLAG_UNMASKED)
    rc = L.hla2_decode_step_mq(_ptr(key_state), _ptr(head_state), _ptr(qd), _ptr(kd), _ptr(vd), _ptr(o), N, Hk,
                               group, d, dv, _ptr(g), int(normalize), _stream_handle(device), ctypes.byref(opts))
    _check("hla2_decode_step_mq", rc)
    return o


def hla3_forward(q, k, v, normalize=False, chunk=64, eps=1e-6, out=None, return_final_state=False):
    """Masked third-order output at gamma = 1 (every factor of A A^T A and the partial product
    of the first two causally masked).  q, k [B,H,n,d]; v [B,H,n,dv] on the GPU, float32 or
    bfloat16.  Returns out [B,H,n,dv] (and with return_final_state the streaming state
    [B,H,state_floats(d, dv)] after the last token, for hla3_decode_step)."""
    L = lib()
    if q.dtype not in _DTYPES or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must all be float32 or all bfloat16")
    if q.device.type != "cuda":
        raise ValueError("q, k, v must be CUDA tensors")
    B, H, n, d = q.shape
    dv = v.shape[-1]
    device = q.device
    qd, kd, vd = (t.contiguous() for t in (q, k, v))
    o = out if out is not None else torch.empty((B, H, n, dv), dtype=q.dtype, device=device)
    sh = _stream_handle(device)
    nbytes = L.hla2_hla3_forward_workspace_bytes(B, H, n, d, dv, chunk, _DTYPES[q.dtype], int(normalize),
                                                 int(return_final_state))
    if nbytes == ctypes.c_size_t(-1).value:
        nbytes = 0
    ws = _workspace(int(nbytes), device, sh)
    fin = torch.empty((B, H, state_floats(d, dv)), dtype=torch.float32, device=device) if return_final_state else None
    opts = Opts(_DTYPES[q.dtype], float(eps), None if ws is None else ws.data_ptr(), int(nbytes), None,
                None if fin is None else fin.data_ptr(), None, 0, 0)
    _check("hla2_hla3_forward", L.hla2_hla3_forward(_ptr(qd), _ptr(kd), _ptr(vd), _ptr(o), B, H, n, d, dv, None,
                                                    int(normalize), chunk, sh, ctypes.byref(opts)))
    return (o, fin) if return_final_state else o


def hla3_decode_step(state, q, k, v, normalize=False, eps=1e-6, out=None):
    """One third-order streaming step (gamma = 1).  state [N,H,state_floats(d, dv)] float32 on
    the GPU, laid out S^K | P^KV | Y | m^K | y, updated in place; q, k [N,H,d]; v [N,H,dv].
    Returns out [N,H,dv]."""
    L = lib()
    if state.device.type != "cuda" or state.dtype != torch.float32 or not state.is_contiguous():
        raise ValueError("state must be a contiguous float32 CUDA tensor")
    device = state.device
    N, H, d = q.shape
    dv = v.shape[-1]
    qd, kd, vd = (_to_device(t, device) for t in (q, k, v))
    o = out if out is not None else torch.empty((N, H, dv), dtype=q.dtype, device=device)
    opts = Opts(_DTYPES[q.dtype], float(eps), None, 0, None, None, None, 0, 0)
    _check("hla2_hla3_decode_step", L.hla2_hla3_decode_step(_ptr(state), _ptr(qd), _ptr(kd), _ptr(vd), _ptr(o), N,
                                                            H, d, dv, int(normalize), _stream_handle(device),
                                                            ctypes.byref(opts)))
    return o


def ahla_backward(q, k, v, dout, gamma=None, chunk=32):
    """Gradients (dq, dk, dv) of the unnormalised AHLA output for upstream dout.  float32 or
    bfloat16 CUDA tensors [B,H,n,d] (d == dv)."""
    L = lib()
    if q.dtype not in _DTYPES or any(t.dtype != q.dtype for t in (k, v, dout)):
        raise TypeError("q, k, v, dout must share a dtype (float32 or bfloat16)")
    B, H, n, d = q.shape
    dv = v.shape[-1]
    device = q.device
    qd, kd, vd, od = (t.contiguous() for t in (q, k, v, dout))
    g = _gamma_tensor(gamma, H, device)
    gq, gk, gv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    sh = _stream_handle(device)
    nbytes = L.hla2_ahla_backward_workspace_bytes(B, H, n, d, dv, chunk, _DTYPES[q.dtype], 0)
    if nbytes == ctypes.c_size_t(-1).value:
        nbytes = 0
    ws = _workspace(int(nbytes), device, sh)
    opts = Opts(_DTYPES[q.dtype], 1e-6, None if ws is None else ws.data_ptr(), int(nbytes), None, None, None, 0, 0)
    _check("hla2_ahla_backward", L.hla2_ahla_backward(_ptr(qd), _ptr(kd), _ptr(vd), _ptr(od), _ptr(gq), _ptr(gk),
                                                      _ptr(gv), B, H, n, d, dv, _ptr(g), 0, chunk, sh,
                                                      ctypes.byref(opts)))
    return gq, gk, gv
