"""GB300-native causal shared-offset sparse attention (libsfa binding).

The compute path is libsfa.so (hand-written sm_103a CUDA, C ABI declared in
include/sfa.h); this package only marshals torch tensors into it.
"""
from ._lib import (LIB_PATH, MAX_RUNGS, SCHED_COPRIME, SCHED_FIXED, SCHED_LINEAR, SFA_BF16,
                   SFA_F32, SfaError)
from .api import (alpha_schedule, backward, backward_int, band_plan, decode_int, forward,
                  forward_int, get_device_status, int_distances, make_desc, offset_histogram,
                  offsets_christoffel, offsets_fib, offsets_pow2, offsets_powerlaw, reach,
                  residue_classes, rope_keys, rope_table, rung_table, status_string, timing_enable,
                  timing_read, workspace_size)

__all__ = [
    "LIB_PATH", "MAX_RUNGS", "SCHED_COPRIME", "SCHED_FIXED", "SCHED_LINEAR", "SFA_BF16",
    "SFA_F32", "SfaError", "alpha_schedule", "backward", "backward_int", "band_plan",
    "decode_int", "forward", "forward_int", "get_device_status", "int_distances", "make_desc", "offsets_christoffel",
    "offset_histogram", "offsets_fib", "offsets_pow2", "offsets_powerlaw", "reach",
    "residue_classes", "rope_keys", "rope_table", "rung_table", "status_string",
    "workspace_size", "timing_enable", "timing_read",
]
