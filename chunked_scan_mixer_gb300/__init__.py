"""GB300 (sm_103a) implementation of masked second-order Higher-order Linear Attention.

The computation lives in the CUDA library built from ``csrc/`` (C ABI in
``include/hla2.h``); ``hla2`` is its Python binding and ``inputs`` draws the seeded
synthetic workloads.
"""
from .hla2 import (HLA2Error, ahla_decode_step, ahla_forward, ahla_state_floats, backward, check_status, decode_step, forward, forward_plan,  # noqa: F401
                   forward_workspace_bytes, lib, state_floats, state_from_compact, state_to_compact)

__version__ = "0.1.0"
