"""Shared test helpers: error metric, oracle adapters, header parsing."""
import os
import re

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hla2.h")

# Parity bars: max|gpu - oracle| / max|oracle|
TOL_F32 = 1e-4
TOL_BF16 = 2e-2


def tol_for(dtype):
    return TOL_F32 if dtype == torch.float32 else TOL_BF16


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.max(np.abs(ref))
    if scale == 0.0:
        return float(np.max(np.abs(got)))
    return float(np.max(np.abs(got - ref)) / scale)


def np64(t):
    """Exact float64 copy of a (possibly bf16) tensor for the oracle."""
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)


def np32(t):
    return t.detach().to("cpu", torch.float32).numpy()


def header_functions():
    """Names of the functions declared in include/hla2.h."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(hla2_[a-z0-9_]+)\s*\(", src)))


def state_part_errs(got, want, d, dv):
    """rel_err of each part (S, C, m, G, h) of packed states [..., d*d + 2*d*dv + 2*d]: a
    part's error is measured against its own scale, so an error in the small parts (m, h)
    is not hidden by the large ones."""
    from oracle import hla2_oracle as O

    g = O.unpack_state(np.asarray(got, dtype=np.float64), d, dv)
    w = O.unpack_state(np.asarray(want, dtype=np.float64), d, dv)
    return {key: rel_err(g[key], w[key]) for key in ("S", "C", "m", "G", "h")}


def assert_state_parts(got, want, d, dv, tol, what=""):
    errs = state_part_errs(got, want, d, dv)
    bad = {k: e for k, e in errs.items() if not e <= tol}
    assert not bad, f"{what} state parts over {tol}: {bad}"
