"""ctypes binding of libsfa (argument marshalling only).

Every step of the attention runs inside libsfa's CUDA kernels; this module
only turns torch tensors into device pointers, allocates outputs with torch
and forwards the call.  If libsfa.so is missing it raises: there is no CPU
fallback.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsfa.so")
DEBUG_LIB_PATH = os.path.join(_PKG, "libsfa_debug.so")  # SIMT kernels with index checks

SFA_F32, SFA_BF16 = 0, 1
SCHED_FIXED, SCHED_LINEAR, SCHED_COPRIME = 0, 1, 2
MAX_RUNGS = 256


class SfaError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = _lib().sfa_status_string(code).decode() if _LIB is not None else str(code)
        super().__init__(f"{where}: {msg} (status {code})")
        self.code = code


class Desc(C.Structure):
    _fields_ = [
        ("B", C.c_int32), ("T", C.c_int32), ("Hq", C.c_int32), ("Hkv", C.c_int32),
        ("D", C.c_int32), ("dtype", C.c_int32), ("W", C.c_int32), ("alpha", C.c_double),
        ("base", C.POINTER(C.c_int32)), ("n_base", C.c_int32),
        ("dist", C.POINTER(C.c_int32)), ("n_dist", C.c_int32),
        ("rope", C.c_void_p), ("k_rot", C.c_void_p),
    ]


_LIB = None
_LOCK = threading.Lock()
_P = C.c_void_p
_I32P = C.POINTER(C.c_int32)

# argument types of every exported entry point (all return int)
SIGNATURES = {
    "sfa_offsets_fib": [C.c_int32, _I32P],
    "sfa_offsets_pow2": [C.c_int32, _I32P],
    "sfa_offsets_christoffel": [C.c_int32, C.c_int32, C.c_int32, _I32P, C.c_int32, _I32P],
    "sfa_alpha_schedule": [C.c_int32, C.c_int32, C.c_int32, C.POINTER(C.c_double)],
    "sfa_rung_table": [_I32P, C.c_int32, C.c_double, C.c_int32, _I32P,
                       C.POINTER(C.c_float), C.POINTER(C.c_float), C.c_int32, _I32P],
    "sfa_int_distances": [_I32P, C.c_int32, _I32P, C.c_int32, _I32P],
    "sfa_band_plan": [_I32P, C.c_int32, C.c_int32, C.c_int32, _I32P, _I32P, _I32P,
                      C.c_int32, _I32P],
    "sfa_rope_table_bytes": [C.c_int32, C.POINTER(C.c_size_t)],
    "sfa_rope_table": [C.c_int32, C.c_double, _P, _P],
    "sfa_workspace_size": [C.POINTER(Desc), C.c_int, C.c_int, C.POINTER(C.c_size_t)],
    "sfa_forward": [C.POINTER(Desc), _P, _P, _P, _P, _P, _P, C.c_size_t, _P],
    "sfa_forward_int": [C.POINTER(Desc), _P, _P, _P, _P, _P, _P, C.c_size_t, _P],
    "sfa_backward": [C.POINTER(Desc), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                     C.c_size_t, _P],
    "sfa_backward_int": [C.POINTER(Desc), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                         C.c_size_t, _P],
    "sfa_get_device_status": [_P, _I32P],
    "sfa_forward_noalloc": [C.POINTER(Desc), _P, _P, _P, _P, _P, _P],
    "sfa_decode_int": [C.POINTER(Desc), _P, _P, _P, _P, _P, _P, _P],
    "sfa_rope_keys": [C.POINTER(Desc), _P, _P, _P],
    "sfa_reach": [_I32P, _I32P, C.c_int32, C.c_int32, _I32P, C.POINTER(C.c_int64)],
    "sfa_residue_classes": [_I32P, C.c_int32, C.c_int32, C.POINTER(C.c_int64)],
    "sfa_offset_histogram": [_I32P, C.c_int32, C.c_int32, C.c_int32, C.POINTER(C.c_int64)],
    "sfa_offsets_powerlaw": [C.POINTER(C.c_double), C.c_int32, C.c_double, C.c_int32,
                             _I32P, C.c_int32, _I32P],
    "sfa_debug_inject": [C.c_int64, C.c_int32],
    "sfa_set_option": [C.c_int32, C.c_int32],
    "sfa_timing_enable": [C.c_int],
    "sfa_timing_read": [C.POINTER(C.c_double), C.POINTER(C.c_int64), C.c_int],
}


def bind(path: str):
    """Load a build of the library (libsfa.so or the bounds-checked
    libsfa_debug.so) with its argument types set; raises if it is missing."""
    if not os.path.exists(path):
        raise RuntimeError(f"{os.path.basename(path)} not built ({path}); run "
                           "`python -m static_offset_sparse_gb300.build`")
    L = C.CDLL(path)
    for name, args in SIGNATURES.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = C.c_int
    L.sfa_status_string.argtypes = [C.c_int]
    L.sfa_status_string.restype = C.c_char_p
    return L


def _lib():
    global _LIB
    if _LIB is not None:
        return _LIB
    with _LOCK:
        if _LIB is None:
            _LIB = bind(LIB_PATH)
    return _LIB


def check(code: int, where: str) -> None:
    if code != 0:
        raise SfaError(code, where)


def i32_array(xs):
    xs = [int(x) for x in xs]
    return (C.c_int32 * max(1, len(xs)))(*xs), len(xs)
