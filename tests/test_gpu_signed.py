"""GPU parity of the integer path with signed (bidirectional) distance sets:
keys i - s for s in the set with 0 <= i - s < T, a negative s reading the
future row i + |s| ("Christoffel-Balanced Sparse Attention": signed offsets
for bidirectional attention).  Forward and backward against the fp64 oracle,
same bounds as the causal parity tests."""
import numpy as np
import pytest

import oracle as o
import sfa_inputs as si
from tolerances import check_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sfa(sfa_lib):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import static_offset_sparse_gb300 as s

    return s


def _check(name, got, want, bf16):
    check_close(name, got, want, bf16)


SETS = {
    "christoffel16_64": o.signed_christoffel_offsets(16, 64),
    "window_pm3": list(range(-3, 4)),
    "mixed": [-40, -17, -5, -1, 0, 1, 2, 8, 13, 29],
    "future_only": [0, -1, -2, -9],
}
SHAPES = [(1, 40, 4, 2), (2, 130, 8, 2), (1, 300, 4, 4), (1, 17, 16, 1)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("name", sorted(SETS))
def test_signed_forward_backward(sfa, dtype, shape, name):
    import torch

    B, T, Hq, Hkv = shape
    dist = SETS[name]
    theta = 0.0 if name == "window_pm3" else 1e4
    x = si.make_qkvdo(B, T, Hq, Hkv, 64, dtype, seed=900 + T + len(dist))
    dev = {n: t.cuda() for n, t in x.items()}
    O, L = sfa.forward_int(dev["q"], dev["k"], dev["v"], dist=dist, rope_theta=theta)
    dq, dk, dv = sfa.backward_int(dev["q"], dev["k"], dev["v"], O, L, dev["do"], dist=dist,
                                  rope_theta=theta)
    torch.cuda.synchronize()
    assert sfa.get_device_status() == 0
    f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()  # noqa: E731
    slots = o.dist_slots(dist)
    Ow, Lw = o.forward(x["q"], x["k"], x["v"], slots, theta)
    gw = o.backward(x["q"], x["k"], x["v"], x["do"], slots, theta)
    bf16 = dtype == "bf16"
    _check("O", f64(O), Ow, bf16)
    assert np.abs(f64(L) - Lw).max() <= (2e-2 if bf16 else 1e-5)
    _check("dQ", f64(dq), gw["dq"], bf16)
    _check("dK", f64(dk), gw["dk"], bf16)
    _check("dV", f64(dv), gw["dv"], bf16)


def test_decode_rejects_future_keys(sfa):
    import torch

    x = si.make_qkvdo(1, 16, 4, 1, 64, "f32", seed=1, with_do=False)
    dev = {n: t.cuda() for n, t in x.items()}
    pos = torch.zeros((1,), dtype=torch.int32, device="cuda")
    with pytest.raises(sfa.SfaError):
        sfa.decode_int(dev["q"][:, :, 0].contiguous(), dev["k"], dev["v"], pos, dist=[-1, 0])
