"""GPU parity: libsfa (through the C ABI) against the fp64 oracle.

Same seeded inputs on both sides; outputs compared element by element.
Tolerances: max-abs 1e-5 for fp32 I/O and 2e-2 for bf16 I/O on O, dQ, dK,
dV; dL/dtheta (and dL/dalpha) within 1e-3 relative for fp32 I/O and within
the random-walk bound of dalpha_tol for bf16 I/O.  A bf16 output cannot be
closer to the exact value than its own rounding, so the bf16 bound is
2e-2 + half a bf16 ulp of the exact value per element (tolerances.check_close).
"""
import math

import numpy as np
import pytest

import oracle as o
import sfa_inputs as si
from tolerances import check_close, check_dalpha_dtheta

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}


@pytest.fixture(scope="module")
def sfa(sfa_lib):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import static_offset_sparse_gb300 as s

    return s


def _dev(x):
    return x.cuda()


def _np(t):
    import torch

    return t.detach().to("cpu", torch.float64).numpy()


def _run_interp(sfa, x, W, alpha, base, theta, backward=True):
    q, k, v, do = (_dev(x[n]) for n in ("q", "k", "v", "do"))
    O, lse = sfa.forward(q, k, v, W=W, alpha=alpha, base=base, rope_theta=theta)
    if not backward:
        return O, lse, None
    g = sfa.backward(q, k, v, O, lse, do, W=W, alpha=alpha, base=base, rope_theta=theta)
    return O, lse, g


def _check(name, got, want, tol, bf16=None):
    if bf16 is None:
        import torch

        bf16 = got.dtype == torch.bfloat16
    check_close(name, _np(got), want, bf16, tol=tol)


SHAPES = [  # B, T, Hq, Hkv
    (1, 1, 8, 2), (1, 2, 4, 1), (2, 3, 1, 1), (1, 17, 8, 2), (2, 65, 4, 1),
    (1, 130, 8, 2), (1, 300, 2, 2), (1, 70, 16, 1), (1, 40, 2, 1), (1, 90, 8, 1),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("W,alpha", [(0, 1.0), (1, 0.77), (8, 1.5), (3, 0.5)])
def test_interp_parity_small(sfa, dtype, shape, W, alpha):
    B, T, Hq, Hkv = shape
    x = si.make_qkvdo(B, T, Hq, Hkv, 64, dtype, seed=100 + T)
    base = o.fib_offsets(12)
    O, lse, g = _run_interp(sfa, x, W, alpha, base, 1e4)
    slots = o.interp_slots(base, alpha, W)
    Ow, Lw = o.forward(x["q"], x["k"], x["v"], slots, 1e4)
    gw = o.backward(x["q"], x["k"], x["v"], x["do"], slots, 1e4, alpha=alpha)
    tol = TOL[dtype]
    _check("O", O, Ow, tol)
    _check("lse", lse, Lw, 1e-5 if dtype == "f32" else 2e-2, bf16=False)
    _check("dQ", g[0], gw["dq"], tol)
    _check("dK", g[1], gw["dk"], tol)
    _check("dV", g[2], gw["dv"], tol)
    da, dt = _np(g[3])
    check_dalpha_dtheta(da, dt, gw, alpha, dtype == "bf16")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("theta", [1e4, 0.0])
@pytest.mark.parametrize("dist_kind", ["fib_round", "christoffel", "pow2", "dense"])
@pytest.mark.parametrize("heads", [(4, 2), (8, 2)])
def test_int_parity_small(sfa, dtype, theta, dist_kind, heads):
    B, T = 2, 97
    Hq, Hkv = heads
    if dist_kind == "fib_round":
        dist = o.int_distances(o.fib_offsets(12), 0.5, 4)
    elif dist_kind == "christoffel":
        dist = o.christoffel_offsets(3, 8) + [11, 13, 16, 21]
    elif dist_kind == "pow2":
        dist = [0] + o.pow2_offsets(8)
    else:
        dist = list(range(T))  # dense causal attention
    x = si.make_qkvdo(B, T, Hq, Hkv, 64, dtype, seed=7)
    q, k, v, do = (_dev(x[n]) for n in ("q", "k", "v", "do"))
    O, lse = sfa.forward_int(q, k, v, dist=dist, rope_theta=theta)
    dq, dk, dv = sfa.backward_int(q, k, v, O, lse, do, dist=dist, rope_theta=theta)
    slots = o.dist_slots(dist)
    Ow, _ = o.forward(x["q"], x["k"], x["v"], slots, theta)
    gw = o.backward(x["q"], x["k"], x["v"], x["do"], slots, theta)
    tol = TOL[dtype]
    _check("O", O, Ow, tol)
    _check("dQ", dq, gw["dq"], tol)
    _check("dK", dk, gw["dk"], tol)
    _check("dV", dv, gw["dv"], tol)


def test_interp_at_integer_alpha_equals_int_path(sfa):
    """At alpha = 1 the interpolation weights are 0: both paths agree."""
    x = si.make_qkvdo(1, 200, 8, 2, 64, "f32", seed=3)
    base = o.fib_offsets(15)
    O1, L1, _ = _run_interp(sfa, x, 8, 1.0, base, 1e4, backward=False)
    q, k, v = (_dev(x[n]) for n in ("q", "k", "v"))
    O2, L2 = sfa.forward_int(q, k, v, dist=o.int_distances(base, 1.0, 8), rope_theta=1e4)
    assert np.abs(_np(O1) - _np(O2)).max() <= 1e-6
    assert np.abs(_np(L1) - _np(L2)).max() <= 1e-6


def test_guard_bands_and_determinism(sfa):
    import torch

    B, T, Hq, Hkv = 2, 77, 8, 2
    x = si.make_qkvdo(B, T, Hq, Hkv, 64, "bf16", seed=5)
    q, k, v, do = (_dev(x[n]) for n in ("q", "k", "v", "do"))
    pad = 4096
    big = {n: torch.full((pad * 2 + t.numel(),), 7.0, dtype=t.dtype, device="cuda")
           for n, t in (("o", q), ("dq", q), ("dk", k), ("dv", v))}
    view = {n: big[n][pad : pad + (q if n in ("o", "dq") else k).numel()].view(
        (q if n in ("o", "dq") else k).shape) for n in big}
    base = o.fib_offsets(15)
    runs = []
    for _ in range(3):
        O, lse = sfa.forward(q, k, v, W=8, alpha=0.83, base=base, o=view["o"])
        dq, dk, dv, dadt = sfa.backward(q, k, v, O, lse, do, W=8, alpha=0.83, base=base,
                                        dq=view["dq"], dk=view["dk"], dv=view["dv"])
        runs.append([t.clone() for t in (O, lse, dq, dk, dv, dadt)])
    for n, b in big.items():
        assert (b[:pad] == 7.0).all() and (b[-pad:] == 7.0).all(), f"{n} guard band overwritten"
    for r in runs[1:]:
        for a_, b_ in zip(runs[0], r):
            assert torch.equal(a_, b_), "run-to-run results differ"
    assert sfa.get_device_status() == 0


def test_errors_leave_outputs_untouched(sfa):
    import torch

    q = torch.zeros((1, 8, 16, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 2, 16, 64), dtype=torch.bfloat16, device="cuda")
    o_ = torch.full_like(q, 3.0)
    with pytest.raises(sfa.SfaError):
        sfa.forward_int(q, k, k, dist=[1, 2], o=o_)  # distance 0 missing
    with pytest.raises(sfa.SfaError):
        sfa.forward(q, k, k, W=-1, alpha=1.0, base=[1, 2], o=o_)
    torch.cuda.synchronize()
    assert (o_ == 3.0).all()


def test_k_rot_reuse_is_bit_identical(sfa):
    """Passing the rotated keys of rope_keys (one rotation per layer) gives the
    same bits as the calls' own rotation, and shrinks their workspaces."""
    import torch

    x = si.make_qkvdo(2, 150, 8, 2, 64, "bf16", seed=61)
    d = {n: t.cuda() for n, t in x.items()}
    base = o.fib_offsets(12)
    kr = sfa.rope_keys(d["k"])
    O1, L1 = sfa.forward(d["q"], d["k"], d["v"], W=8, alpha=0.9, base=base)
    O2, L2 = sfa.forward(d["q"], d["k"], d["v"], W=8, alpha=0.9, base=base, k_rot=kr)
    g1 = sfa.backward(d["q"], d["k"], d["v"], O1, L1, d["do"], W=8, alpha=0.9, base=base)
    g2 = sfa.backward(d["q"], d["k"], d["v"], O2, L2, d["do"], W=8, alpha=0.9, base=base, k_rot=kr)
    torch.cuda.synchronize()
    assert torch.equal(O1, O2) and torch.equal(L1, L2)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)
    d1 = sfa.make_desc(d["q"], d["k"], W=8, alpha=0.9, base=base)
    d2 = sfa.make_desc(d["q"], d["k"], W=8, alpha=0.9, base=base, k_rot=kr)
    assert sfa.workspace_size(d2, True, False) == 0 < sfa.workspace_size(d1, True, False)
    assert sfa.workspace_size(d2, True, True) < sfa.workspace_size(d1, True, True)


@pytest.mark.parametrize("B,T,Hq,Hkv", [(2, 200, 16, 2), (1, 256, 8, 1), (1, 333, 32, 8)])
def test_rung_kernels_groups_of_four_heads(sfa, B, T, Hq, Hkv):
    """G = 8 and 16: the rung kernels run one CTA row per group of four query
    heads (reading KV head group / (G / 4)) and the key side sums the groups;
    interpolated (with dL/dalpha) and integer paths against the oracle."""
    base = o.fib_offsets(15)
    x = si.make_qkvdo(B, T, Hq, Hkv, 64, "bf16", seed=300 + Hq + T)
    alpha = 0.83
    O, L, g = _run_interp(sfa, x, 8, alpha, base, 1e4)
    slots = o.interp_slots(base, alpha, 8)
    Ow, Lw = o.forward(x["q"], x["k"], x["v"], slots, 1e4)
    gw = o.backward(x["q"], x["k"], x["v"], x["do"], slots, 1e4, alpha=alpha)
    _check("O", O, Ow, 2e-2)
    _check("LSE", L, Lw, 2e-2, bf16=False)
    for name, got, key in (("dQ", g[0], "dq"), ("dK", g[1], "dk"), ("dV", g[2], "dv")):
        _check(name, got, gw[key], 2e-2)
    da, dt = _np(g[3])
    check_dalpha_dtheta(da, dt, gw, alpha, True)
    dist = sorted(set(range(9)) | set(o.fib_offsets(15)))
    q, k, v, do = (_dev(x[n]) for n in ("q", "k", "v", "do"))
    Oi, Li = sfa.forward_int(q, k, v, dist=dist)
    gi = sfa.backward_int(q, k, v, Oi, Li, do, dist=dist)
    si_ = o.dist_slots(dist)
    Ow, _ = o.forward(x["q"], x["k"], x["v"], si_, 1e4)
    gw = o.backward(x["q"], x["k"], x["v"], x["do"], si_, 1e4)
    _check("O int", Oi, Ow, 2e-2)
    for name, got, key in (("dQ int", gi[0], "dq"), ("dK int", gi[1], "dk"), ("dV int", gi[2], "dv")):
        _check(name, got, gw[key], 2e-2)
    assert sfa.get_device_status() == 0


@pytest.mark.parametrize("W,T,Hq", [(10, 70, 8), (12, 300, 8), (12, 129, 16), (9, 41, 4)])
def test_rung_kernels_wide_window(sfa, W, T, Hq):
    """Windows of 9 to 13 distances on the rung kernels: the key side stages a
    window chunk of up to 9 distances (at G = 4 as two groups, its q~ slab with
    the records, then its dO slab), so W = 10 and 12 take two chunks; ragged T,
    interpolated (with dL/dalpha) and integer paths, element by element."""
    base = o.fib_offsets(15)
    x = si.make_qkvdo(1, T, Hq, 2 if Hq > 4 else 1, 64, "bf16", seed=400 + W + T)
    alpha = 0.77
    O, L, g = _run_interp(sfa, x, W, alpha, base, 1e4)
    slots = o.interp_slots(base, alpha, W)
    Ow, Lw = o.forward(x["q"], x["k"], x["v"], slots, 1e4)
    gw = o.backward(x["q"], x["k"], x["v"], x["do"], slots, 1e4, alpha=alpha)
    _check("O", O, Ow, 2e-2)
    _check("LSE", L, Lw, 2e-2, bf16=False)
    for name, got, key in (("dQ", g[0], "dq"), ("dK", g[1], "dk"), ("dV", g[2], "dv")):
        _check(name, got, gw[key], 2e-2)
    da, dt = _np(g[3])
    check_dalpha_dtheta(da, dt, gw, alpha, True)
    dist = sorted(set(range(W + 1)) | {round(alpha * f) for f in base})
    q, k, v, do = (_dev(x[n]) for n in ("q", "k", "v", "do"))
    Oi, Li = sfa.forward_int(q, k, v, dist=dist)
    gi = sfa.backward_int(q, k, v, Oi, Li, do, dist=dist)
    si_ = o.dist_slots(dist)
    Ow, _ = o.forward(x["q"], x["k"], x["v"], si_, 1e4)
    gw = o.backward(x["q"], x["k"], x["v"], x["do"], si_, 1e4)
    _check("O int", Oi, Ow, 2e-2)
    for name, got, key in (("dQ int", gi[0], "dq"), ("dK int", gi[1], "dk"), ("dV int", gi[2], "dv")):
        _check(name, got, gw[key], 2e-2)
    assert sfa.get_device_status() == 0
