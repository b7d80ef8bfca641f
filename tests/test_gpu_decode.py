"""GPU parity of the integer-path decode step (one query per sequence against
a key/value cache) with the fp64 oracle.

The oracle's decode (pinned to the forward's row pos[b] of the prefix)
gives the expected rows.  Same seeded inputs on both sides;
bounds as for the forward: 1e-5 (fp32 I/O) and 2e-2 plus half a bf16 ulp of
the exact value (bf16).
"""
import numpy as np
import pytest

import oracle as o
import sfa_inputs as si
from tolerances import check_close

pytestmark = pytest.mark.gpu

FIB = o.fib_offsets(15)


@pytest.fixture(scope="module")
def sfa(sfa_lib):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import static_offset_sparse_gb300 as s

    return s


def _expected(q, k, v, pos, dist, theta):
    return o.decode(q, k, v, pos, dist, theta)


def _check(name, got, want, bf16):
    check_close(name, got, want, bf16)


CASES = [  # B, T (cache), Hq, Hkv, dist, positions, theta
    (3, 200, 8, 2, "fib1", [0, 57, 199], 1e4),
    (4, 130, 4, 4, "christoffel16_64", [129, 7, 64, 1], 1e4),
    (2, 70, 16, 1, "fib05", [69, 3], 0.0),
    (5, 40, 2, 1, "window", [39, 0, 12, 38, 20], 1e4),
    (2, 1100, 4, 2, "christoffel128_1024", [1099, 700], 1e4),
]


def _dist(name):
    if name == "fib1":
        return o.int_distances(FIB, 1.0, 8)
    if name == "fib05":
        return o.int_distances(FIB, 0.5, 3)
    if name == "window":
        return list(range(0, 13))
    m, k = (int(x) for x in name[len("christoffel"):].split("_"))
    return o.christoffel_offsets(m, k, include_zero=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_decode_matches_oracle(sfa, dtype, case):
    import torch

    B, T, Hq, Hkv, dname, pos, theta = CASES[case]
    dist = _dist(dname)
    x = si.make_qkvdo(B, T, Hq, Hkv, 64, dtype, seed=500 + case, with_do=False)
    q_dec = x["q"][:, :, -1].contiguous()  # one query row per (b, head)
    dev = {n: t.cuda() for n, t in x.items()}
    posd = torch.tensor(pos, dtype=torch.int32, device="cuda")
    O, L = sfa.decode_int(q_dec.cuda(), dev["k"], dev["v"], posd, dist=dist, rope_theta=theta)
    torch.cuda.synchronize()
    assert sfa.get_device_status() == 0
    f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()  # noqa: E731
    Ow, Lw = _expected(f64(q_dec), f64(x["k"]), f64(x["v"]), pos, dist, theta)
    _check("O", f64(O), Ow, dtype == "bf16")
    lse_tol = 1e-5 if dtype == "f32" else 2e-2
    assert np.abs(f64(L) - Lw).max() <= lse_tol


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_both_kernels(sfa, dtype):
    """Steps of more than 1024 heads run the register kernel, smaller steps the
    staged one: B = 130 sequences x 8 heads against the oracle, and its first
    three sequences bit for bit against a three-sequence call."""
    import torch

    B, T, Hq, Hkv = 130, 64, 8, 2
    dist = o.int_distances(FIB, 1.0, 8)
    x = si.make_qkvdo(B, T, Hq, Hkv, 64, dtype, seed=91, with_do=False)
    rng = np.random.default_rng(5)
    pos = [int(p) for p in rng.integers(0, T, size=B)]
    q_dec = x["q"][:, :, -1].contiguous().cuda()
    k, v = x["k"].cuda(), x["v"].cuda()
    posd = torch.tensor(pos, dtype=torch.int32, device="cuda")
    O, L = sfa.decode_int(q_dec, k, v, posd, dist=dist)
    O3, L3 = sfa.decode_int(q_dec[:3].contiguous(), k[:3].contiguous(), v[:3].contiguous(),
                            posd[:3].contiguous(), dist=dist)
    torch.cuda.synchronize()
    assert sfa.get_device_status() == 0
    assert torch.equal(O[:3], O3) and torch.equal(L[:3], L3)
    f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()  # noqa: E731
    Ow, Lw = _expected(f64(q_dec), f64(x["k"]), f64(x["v"]), pos, dist, 1e4)
    _check("O", f64(O), Ow, dtype == "bf16")
    assert np.abs(f64(L) - Lw).max() <= (1e-5 if dtype == "f32" else 2e-2)


def test_decode_equals_forward_int_row(sfa):
    """Decode at position t reproduces row t of the integer forward (same
    caches, q placed at t)."""
    import torch

    B, T, Hq, Hkv = 2, 96, 8, 2
    dist = o.int_distances(FIB, 1.0, 8)
    x = si.make_qkvdo(B, T, Hq, Hkv, 64, "f32", seed=77, with_do=False)
    dev = {n: t.cuda() for n, t in x.items()}
    Of, Lf = sfa.forward_int(dev["q"], dev["k"], dev["v"], dist=dist)
    for t in (0, 13, 95):
        posd = torch.full((B,), t, dtype=torch.int32, device="cuda")
        Od, Ld = sfa.decode_int(dev["q"][:, :, t].contiguous(), dev["k"], dev["v"], posd, dist=dist)
        assert torch.allclose(Od, Of[:, :, t], atol=2e-6, rtol=0)
        assert torch.allclose(Ld, Lf[:, :, t], atol=2e-6, rtol=0)


def test_decode_bad_position_sets_status(sfa):
    """A position outside the cache is skipped and reported, not read."""
    import torch

    B, T = 2, 32
    x = si.make_qkvdo(B, T, 4, 1, 64, "f32", seed=3, with_do=False)
    dev = {n: t.cuda() for n, t in x.items()}
    posd = torch.tensor([5, T], dtype=torch.int32, device="cuda")
    O, _ = sfa.decode_int(dev["q"][:, :, 0].contiguous(), dev["k"], dev["v"], posd, dist=[0, 1, 2])
    assert sfa.get_device_status() == 6  # SFA_ERR_DEVICE_BOUNDS
    assert sfa.get_device_status() == 0  # read clears it
    Ow, _ = _expected(x["q"][:1, :, 0].double().numpy(), x["k"][:1].double().numpy(),
                      x["v"][:1].double().numpy(), [5], [0, 1, 2], 1e4)
    _check("O[0]", O[:1].double().cpu().numpy(), Ow, False)
