"""The bounds-checked build of the SIMT kernels (libsfa_debug.so) on the GPU.

libsfa_debug.so is libsfa.so with the SIMT kernels (fp32 I/O, and bf16
calls with one or two query heads per KV head or signed sets that have no
band plan)
compiled with SFA_DEBUG_BOUNDS: every row index they form, into the sequence
and into their shared-memory slabs, is range-checked; a bad one is recorded
as SFA_ERR_DEVICE_BOUNDS and its access skipped, with no trap.  These cases
run the SIMT paths through that build: the status word must stay clear and
the results must match the oracle as they do for the release build.
"""
import ctypes as C
import os

import numpy as np
import pytest

import oracle as o
import sfa_inputs as si
from tolerances import check_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from static_offset_sparse_gb300 import _lib, build

    if not os.path.exists(_lib.DEBUG_LIB_PATH):
        build.build()
    return _lib.bind(_lib.DEBUG_LIB_PATH)


CASES = [  # B, T, Hq, Hkv, dtype, kind
    (1, 150, 8, 2, "f32", "interp"),    # fp32 I/O: SIMT, G = 4
    (2, 97, 2, 1, "bf16", "interp"),    # G = 2 bf16: SIMT
    (1, 70, 16, 1, "f32", "int"),       # G = 16 fp32
    (2, 90, 4, 4, "f32", "signed"),     # signed (bidirectional) set, fp32: SIMT
]


@pytest.mark.parametrize("case", CASES)
def test_simt_paths_under_bounds_checks(dbg, case):
    import torch

    import static_offset_sparse_gb300 as sfa

    B, T, Hq, Hkv, dtype, kind = case
    x = si.make_qkvdo(B, T, Hq, Hkv, 64, dtype, seed=900 + T)
    d = {n: t.cuda() for n, t in x.items()}
    base = o.fib_offsets(12)
    if kind == "interp":
        W, alpha = 5, 0.83
        desc = sfa.make_desc(d["q"], d["k"], W=W, alpha=alpha, base=base)
        slots = o.interp_slots(base, alpha, W)
        fwd, bwd, interp = dbg.sfa_forward, dbg.sfa_backward, 1
    else:
        dist = (o.int_distances(base, 1.0, 4) if kind == "int"
                else sorted(set(o.signed_christoffel_offsets(16, 64)) | {0}))
        desc = sfa.make_desc(d["q"], d["k"], dist=dist)
        slots = o.dist_slots(dist)
        fwd, bwd, interp = dbg.sfa_forward_int, dbg.sfa_backward_int, 0
    P = lambda t: C.c_void_p(t.data_ptr())  # noqa: E731
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    n = C.c_size_t(0)
    assert dbg.sfa_workspace_size(C.byref(desc), interp, 1, C.byref(n)) == 0
    ws = torch.zeros(max(1, n.value), dtype=torch.uint8, device="cuda")
    O = torch.empty_like(d["q"])
    L = torch.empty((B, Hq, T), dtype=torch.float32, device="cuda")
    assert fwd(C.byref(desc), P(d["q"]), P(d["k"]), P(d["v"]), P(O), P(L), P(ws), n.value, stream) == 0
    dq, dk, dv = torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"])
    if interp:
        dadt = torch.zeros(2, dtype=torch.float64, device="cuda")
        rc = bwd(C.byref(desc), P(d["q"]), P(d["k"]), P(d["v"]), P(O), P(L), P(d["do"]), P(dq),
                 P(dk), P(dv), P(dadt), P(ws), n.value, stream)
    else:
        rc = bwd(C.byref(desc), P(d["q"]), P(d["k"]), P(d["v"]), P(O), P(L), P(d["do"]), P(dq),
                 P(dk), P(dv), P(ws), n.value, stream)
    assert rc == 0
    torch.cuda.synchronize()
    status = C.c_int32(-1)
    assert dbg.sfa_get_device_status(stream, C.byref(status)) == 0
    assert status.value == 0, "a bounds check fired"
    Ow, _ = o.forward(x["q"], x["k"], x["v"], slots, 1e4)
    gw = o.backward(x["q"], x["k"], x["v"], x["do"], slots, 1e4)
    f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()  # noqa: E731
    bf16 = dtype == "bf16"
    check_close("O", f64(O), Ow, bf16)
    check_close("dQ", f64(dq), gw["dq"], bf16)
    check_close("dK", f64(dk), gw["dk"], bf16)
    check_close("dV", f64(dv), gw["dv"], bf16)
