"""The bounded-wait failure path of the TMA-staged kernels, on the GPU.

Every mbarrier wait of those kernels is bounded.  Through the C ABI's test
injection (sfa_debug_inject) CTA (0, 0) of the rung forward never issues the
loads of one staged group, so that stage's barrier never completes, and the
wait limit is shortened to 1e5 SM cycles.  The call must record
SFA_ERR_TIMEOUT in the device status word and return without hanging; the
status read clears the word; with the injection off, the next calls on the
same stream and context match the oracle again.  Nothing faults or traps:
the failure is a flag that nothing sets, and the wait gives up on its own.
"""
import ctypes as C

import pytest

import oracle as o
import sfa_inputs as si
from tolerances import check_close

pytestmark = pytest.mark.gpu

SFA_ERR_TIMEOUT = 5


@pytest.fixture(scope="module")
def sfa(sfa_lib):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import static_offset_sparse_gb300 as s

    return s


# bf16, G = 4: the rung tensor-core kernels.  CTA (0, 0) (positions 0..15)
# stages two window chunks at W = 12, alpha = 0.9 (skipping chunk 1, loaded
# before the loop), and at W = 0, alpha = 0.5 one chunk and four rung pairs
# (skipping pair 2, loaded by the in-loop refill)
@pytest.mark.parametrize("W,alpha,skip_group", [(12, 0.9, 1), (0, 0.5, 3)])
def test_wait_times_out_and_context_recovers(sfa, sfa_lib, W, alpha, skip_group):
    import torch

    B, T, Hq, Hkv = 1, 160, 8, 2
    base = o.fib_offsets(15)
    xh = si.make_qkvdo(B, T, Hq, Hkv, 64, "bf16", seed=515)
    x = {n: t.cuda() for n, t in xh.items()}
    assert sfa.get_device_status() == 0
    try:
        assert sfa_lib.sfa_debug_inject(C.c_int64(100000), C.c_int32(skip_group)) == 0
        sfa.forward(x["q"], x["k"], x["v"], W=W, alpha=alpha, base=base)
        torch.cuda.synchronize()
    finally:
        assert sfa_lib.sfa_debug_inject(C.c_int64(0), C.c_int32(-1)) == 0
    assert sfa.get_device_status() == SFA_ERR_TIMEOUT
    assert sfa.get_device_status() == 0  # the read cleared the word

    # the context is intact: a normal forward and backward match the oracle
    O, lse = sfa.forward(x["q"], x["k"], x["v"], W=W, alpha=alpha, base=base)
    dq, dk, dv, _ = sfa.backward(x["q"], x["k"], x["v"], O, lse, x["do"], W=W, alpha=alpha,
                                 base=base)
    torch.cuda.synchronize()
    assert sfa.get_device_status() == 0
    slots = o.interp_slots(base, alpha, W)
    Ow, _ = o.forward(xh["q"], xh["k"], xh["v"], slots, 1e4)
    gw = o.backward(xh["q"], xh["k"], xh["v"], xh["do"], slots, 1e4, alpha=alpha)
    f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()  # noqa: E731
    check_close("O", f64(O), Ow, True)
    check_close("dQ", f64(dq), gw["dq"], True)
    check_close("dK", f64(dk), gw["dk"], True)
    check_close("dV", f64(dv), gw["dv"], True)


def test_inject_rejects_bad_arguments(sfa_lib):
    assert sfa_lib.sfa_debug_inject(C.c_int64(-1), C.c_int32(-1)) == 1
    assert sfa_lib.sfa_debug_inject(C.c_int64(0), C.c_int32(-2)) == 1
    assert sfa_lib.sfa_debug_inject(C.c_int64(0), C.c_int32(-1)) == 0
