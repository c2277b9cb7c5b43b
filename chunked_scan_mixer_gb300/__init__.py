"""GB300 (sm_103a) implementation of masked second-order Higher-order Linear Attention.

The computation lives in the CUDA library built from ``csrc/`` (C ABI in
``include/hla2.h``); ``hla2`` is its Python binding and ``inputs`` draws the seeded
synthetic workloads.
"""
from .hla2 import (HLA2Error, ahla_backward, ahla_decode_step, ahla_forward, ahla_state_floats, backward, check_status,  # noqa: F401
                   decode_step, decode_step_mq, forward, forward_plan, forward_workspace_bytes, hla3_decode_step, hla3_forward, lib,
                   mq_head_state_floats, mq_merge_state, mq_split_state, state_floats, state_from_compact,
                   state_to_compact)

__version__ = "0.1.0"
