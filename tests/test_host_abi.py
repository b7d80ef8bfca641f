"""CPU tests of libsfa: exported symbols and the host-side builders.

The builders are compared bit for bit with the oracle's own, independently
written builders; no GPU is used.
"""
import ctypes as C
import os
import re

import numpy as np
import pytest

import oracle as o

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    txt = open(os.path.join(ROOT, "include", "sfa.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(sfa_\w+)\s*\(", txt)))


def test_exports_every_declared_symbol(sfa_lib):
    names = _declared()
    assert len(names) >= 15
    for n in names:
        assert hasattr(sfa_lib, n), n


def test_bounds_checked_build_exports_the_same_symbols(sfa_lib):
    """libsfa_debug.so (SIMT kernels with index checks) is a drop-in build of
    the same C ABI; loading it binds every declared entry point."""
    from static_offset_sparse_gb300 import _lib, build

    if not os.path.exists(_lib.DEBUG_LIB_PATH):
        build.build()
    dbg = _lib.bind(_lib.DEBUG_LIB_PATH)
    for n in _declared():
        assert hasattr(dbg, n), n
    out = (C.c_int32 * 15)()
    assert dbg.sfa_offsets_fib(15, out) == 0 and out[14] == 987


def test_offsets_match_oracle(sfa_lib):
    import static_offset_sparse_gb300 as s

    for K in (1, 2, 15, 40):
        assert s.offsets_fib(K) == o.fib_offsets(K)
    for K in (1, 11, 31):
        assert s.offsets_pow2(K) == o.pow2_offsets(K)
    for m, k in [(128, 1024), (64, 512), (3, 8), (5, 13), (7, 12), (1, 1), (999, 1000), (1, 4097)]:
        for z in (True, False):
            assert s.offsets_christoffel(m, k, z) == o.christoffel_offsets(m, k, z), (m, k, z)


def test_schedules_match_oracle(sfa_lib):
    import static_offset_sparse_gb300 as s

    for kind in (s.SCHED_FIXED, s.SCHED_LINEAR, s.SCHED_COPRIME):
        for L, S in ((16, 7), (5, 3), (1, 1)):
            assert s.alpha_schedule(L, kind, S) == o.alpha_schedule(L, kind, S)


@pytest.mark.parametrize("alpha", [0.5, 1.0, 1.5, 0.5 + 5 / 15, 0.77, 0.5 + 13 / 15])
@pytest.mark.parametrize("W", [0, 6, 8, 12])
def test_rung_table_matches_oracle(sfa_lib, alpha, W):
    import static_offset_sparse_gb300 as s

    for base in (o.fib_offsets(15), o.pow2_offsets(11)):
        c, w, f = s.rung_table(base, alpha, W)
        want = sorted(o.interp_rungs(base, alpha, W), key=lambda r: r["c"])
        assert c == [r["c"] for r in want]
        assert w == [float(np.float32(r["w"])) for r in want]
        assert f == [r["f"] for r in want]


def test_int_distances_match_oracle(sfa_lib):
    import static_offset_sparse_gb300 as s

    for alpha in (0.5, 1.0, 1.5):
        d = o.int_distances(o.fib_offsets(), alpha, 8)
        shuffled = list(reversed(d)) + d[:3]
        assert s.int_distances(shuffled) == d


def test_argument_errors(sfa_lib):
    L = sfa_lib
    out = (C.c_int32 * 64)()
    n = C.c_int32(0)
    assert L.sfa_offsets_fib(0, out) == 1
    assert L.sfa_offsets_fib(41, out) == 1
    assert L.sfa_offsets_pow2(32, out) == 1
    assert L.sfa_offsets_christoffel(5, 4, 1, out, 64, C.byref(n)) == 1
    assert L.sfa_offsets_christoffel(128, 1024, 1, out, 64, C.byref(n)) == 3 and n.value == 129
    sched = (C.c_double * 16)()
    assert L.sfa_alpha_schedule(16, 2, 4, sched) == 1  # gcd(4, 16) != 1
    assert L.sfa_alpha_schedule(16, 9, 7, sched) == 1
    base = (C.c_int32 * 2)(1, 0)
    assert L.sfa_rung_table(base, 2, 1.0, 0, None, None, None, 8, C.byref(n)) == 1
    assert L.sfa_rung_table(base, 1, -1.0, 0, None, None, None, 8, C.byref(n)) == 1
    assert L.sfa_status_string(0) == b"ok"


def test_descriptor_validation_without_gpu(sfa_lib):
    """Shape checks run on the host before anything touches the device."""
    from static_offset_sparse_gb300._lib import Desc

    size = C.c_size_t(0)
    d = Desc()
    d.B, d.T, d.Hq, d.Hkv, d.D, d.dtype, d.W, d.alpha = 1, 16, 8, 2, 64, 1, 8, 1.0
    assert sfa_lib.sfa_workspace_size(C.byref(d), 1, 1, C.byref(size)) == 0 and size.value > 0
    d.D = 128
    assert sfa_lib.sfa_workspace_size(C.byref(d), 1, 1, C.byref(size)) == 2
    d.D, d.Hq = 64, 6  # G = 3 not a power of two
    assert sfa_lib.sfa_workspace_size(C.byref(d), 1, 1, C.byref(size)) == 2
    d.Hq, d.dtype = 8, 7
    assert sfa_lib.sfa_workspace_size(C.byref(d), 1, 1, C.byref(size)) == 1
    d.dtype = 1
    dist = (C.c_int32 * 2)(3, 5)  # distance 0 missing: a query could have no key
    d.dist, d.n_dist = C.cast(dist, C.POINTER(C.c_int32)), 2
    assert sfa_lib.sfa_workspace_size(C.byref(d), 0, 1, C.byref(size)) == 1


def test_empty_and_oversized_shapes_are_rejected_on_the_host(sfa_lib):
    """Empty inputs (a zero extent) and shapes past the grid limits are
    refused by the shape check, before any pointer or the device is touched:
    the compute entry points return the error with null buffers on a machine
    without a GPU.  The largest accepted shape still sizes its workspace."""
    from static_offset_sparse_gb300._lib import Desc

    size = C.c_size_t(0)
    null = C.c_void_p(0)

    def desc(B=1, T=16, Hq=8, Hkv=2):
        d = Desc()
        d.B, d.T, d.Hq, d.Hkv, d.D, d.dtype, d.W, d.alpha = B, T, Hq, Hkv, 64, 1, 8, 1.0
        return d

    for kw in ({"B": 0}, {"T": 0}, {"Hq": 0, "Hkv": 0}, {"Hkv": 0}, {"T": -5}):
        d = desc(**kw)
        assert sfa_lib.sfa_workspace_size(C.byref(d), 1, 1, C.byref(size)) == 1, kw
        assert sfa_lib.sfa_forward(C.byref(d), null, null, null, null, null, null, 0, null) == 1, kw
        assert sfa_lib.sfa_backward(C.byref(d), null, null, null, null, null, null, null, null,
                                    null, null, null, 0, null) == 1, kw
    for kw in ({"T": (1 << 24) + 1}, {"B": 65536, "Hq": 4, "Hkv": 1}, {"B": 32768, "Hkv": 2}):
        d = desc(**kw)
        assert sfa_lib.sfa_workspace_size(C.byref(d), 1, 1, C.byref(size)) == 2, kw
        assert sfa_lib.sfa_forward(C.byref(d), null, null, null, null, null, null, 0, null) == 2, kw
    # G = 8 on the rung kernels: one grid row per group of four query heads, so
    # B Hq / 4 <= 65535 (B Hkv alone would allow twice as many sequences)
    for B, rc in ((16383, 0), (16384, 2)):
        d = desc(B=B, T=16, Hq=16, Hkv=2)
        assert sfa_lib.sfa_workspace_size(C.byref(d), 1, 1, C.byref(size)) == rc, B
        assert sfa_lib.sfa_workspace_size(C.byref(d), 1, 0, C.byref(size)) == rc, B
    d = desc(B=1, T=1 << 24)
    assert sfa_lib.sfa_workspace_size(C.byref(d), 1, 1, C.byref(size)) == 0
    assert size.value > (1 << 24) * 8 * 8  # at least the per-query records of the key side


def test_int_distances_accept_signed_sets(sfa_lib):
    import static_offset_sparse_gb300 as s
    from static_offset_sparse_gb300 import SfaError

    d = [5, -3, 0, -3, 1, -40, 5]
    assert s.int_distances(d) == sorted(set(d))
    with pytest.raises(SfaError):
        s.int_distances([0, 1 << 30])
