"""The allocation-free forward (sfa_forward_noalloc) against sfa_forward and
the oracle.

sfa_forward_noalloc serves callers that cannot allocate device memory: it
keeps the forward's scratch in a fixed device array inside the library.
Called through the C ABI twice in a row, it must give the results of
sfa_forward (caller workspace) and of the fp64 oracle within the parity
tests' bf16 bound, and it must refuse a problem whose scratch exceeds the
array.  This file is named to be collected last.
"""
import ctypes as C

import numpy as np
import pytest

import oracle as o
import sfa_inputs as si
from tolerances import bf16_bound, check_close

pytestmark = pytest.mark.gpu


def test_forward_noalloc_matches_forward(sfa_lib):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import static_offset_sparse_gb300 as s

    B, T, Hq, Hkv, W, alpha = 2, 200, 8, 2, 8, 0.77  # bf16 with G = 4: the kernel that uses scratch
    base = o.fib_offsets(15)
    xh = si.make_qkvdo(B, T, Hq, Hkv, 64, "bf16", seed=77)
    x = {n: t.cuda() for n, t in xh.items()}
    Ow, Lw = o.forward(xh["q"], xh["k"], xh["v"], o.interp_slots(base, alpha, W), 1e4)
    O_ref, L_ref = s.forward(x["q"], x["k"], x["v"], W=W, alpha=alpha, base=base)
    desc = s.make_desc(x["q"], x["k"], W=W, alpha=alpha, base=base)
    assert s.workspace_size(desc, True, False) > 0
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    ref = O_ref.double().cpu().numpy()
    lim = bf16_bound(ref)
    for _ in range(2):
        O = torch.full_like(x["q"], float("nan"))
        L = torch.full((B, Hq, T), float("nan"), dtype=torch.float32, device="cuda")
        rc = sfa_lib.sfa_forward_noalloc(C.byref(desc), C.c_void_p(x["q"].data_ptr()),
                                         C.c_void_p(x["k"].data_ptr()), C.c_void_p(x["v"].data_ptr()),
                                         C.c_void_p(O.data_ptr()), C.c_void_p(L.data_ptr()), stream)
        assert rc == 0, s.status_string(rc)
        torch.cuda.synchronize()
        got = O.double().cpu().numpy()
        assert (np.abs(got - ref) <= lim).all()
        assert (torch.abs(L - L_ref) <= 2e-2).all()
        check_close("O vs oracle", got, Ow, True)
        check_close("LSE vs oracle", L.double().cpu().numpy(), Lw, False, tol=2e-2)
    assert s.get_device_status() == 0

    # a problem whose scratch is larger than the array is refused up front
    from static_offset_sparse_gb300._lib import Desc

    big = Desc()
    C.pointer(big)[0] = desc  # same keys and RoPE table pointer, then a larger shape
    big.B, big.T = 64, 1024  # 64 * 2 * 1024 rows of K' = 16 MiB > SFA_STATIC_WS_BYTES
    rc = sfa_lib.sfa_forward_noalloc(C.byref(big), C.c_void_p(x["q"].data_ptr()),
                                     C.c_void_p(x["k"].data_ptr()), C.c_void_p(x["v"].data_ptr()),
                                     C.c_void_p(O_ref.data_ptr()), C.c_void_p(L_ref.data_ptr()), stream)
    assert rc == 3  # SFA_ERR_CAPACITY
