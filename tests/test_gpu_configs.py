"""GPU parity at the benchmark configurations' full sizes.

Each configuration runs at its real shape through the same entry points the
benchmark calls.  The oracle checks sampled (batch, KV head) units element by
element (the units are independent); dL/dalpha and dL/dtheta, which sum over
the whole batch, are checked against the oracle over every unit for one
config-2 layer (the kink layer alpha = 0.5 + 5/15).
"""
import numpy as np
import pytest

import oracle as o
import sfa_inputs as si
from tolerances import check_close, check_dalpha_dtheta

pytestmark = pytest.mark.gpu

FIB = o.fib_offsets(15)


@pytest.fixture(scope="module")
def sfa(sfa_lib):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import static_offset_sparse_gb300 as s

    return s


def _np(t):
    import torch

    return t.detach().to("cpu", torch.float64).numpy()


def _close(name, got, want, bf16, tol=None):
    check_close(name, got, want, bf16, tol=tol)


def _sampled(sfa, x, pairs, slots, theta, fwd, bwd, bf16, check_bwd=True):
    dev = {n: t.cuda() for n, t in x.items()}
    O, lse = fwd(dev)
    Ow, Lw = o.forward(x["q"], x["k"], x["v"], slots, theta, rows=pairs)
    G = x["q"].shape[1] // x["k"].shape[1]
    for b, g in pairs:
        hs = slice(g * G, (g + 1) * G)
        _close(f"O[{b},{g}]", _np(O)[b, hs], Ow[b, hs], bf16)
        _close(f"lse[{b},{g}]", _np(lse)[b, hs], Lw[b, hs], False, tol=2e-2 if bf16 else 1e-5)
    if not check_bwd:
        return O, lse, None
    grads = bwd(dev, O, lse)
    gw = o.backward(x["q"], x["k"], x["v"], x["do"], slots, theta, rows=pairs)
    for b, g in pairs:
        hs = slice(g * G, (g + 1) * G)
        _close(f"dQ[{b},{g}]", _np(grads[0])[b, hs], gw["dq"][b, hs], bf16)
        _close(f"dK[{b},{g}]", _np(grads[1])[b, g], gw["dk"][b, g], bf16)
        _close(f"dV[{b},{g}]", _np(grads[2])[b, g], gw["dv"][b, g], bf16)
    return O, lse, grads


def test_config1_fp32_full(sfa):
    """B=1, T=1024, 8/2 heads, W=8, alpha=1, Fibonacci K=15, fp32, seed 0."""
    x = si.make_qkvdo(1, 1024, 8, 2, 64, "f32", seed=0)
    slots = o.interp_slots(FIB, 1.0, 8)
    fwd = lambda d: sfa.forward(d["q"], d["k"], d["v"], W=8, alpha=1.0, base=FIB)
    bwd = lambda d, O, L: sfa.backward(d["q"], d["k"], d["v"], O, L, d["do"], W=8, alpha=1.0, base=FIB)
    _, _, g = _sampled(sfa, x, [(0, 0), (0, 1)], slots, 1e4, fwd, bwd, False)
    gw = o.backward(x["q"], x["k"], x["v"], x["do"], slots, 1e4, alpha=1.0)
    da, dt = _np(g[3])
    # at alpha = 1 (theta = 0) dtheta = dalpha (1 - 0.5)(1.5 - 1) = dalpha / 4, not zero
    assert abs(gw["dtheta"] - 0.25 * gw["dalpha"]) <= 1e-12 * abs(gw["dalpha"])
    assert abs(da - gw["dalpha"]) <= 1e-3 * abs(gw["dalpha"])
    assert abs(dt - gw["dtheta"]) <= 1e-3 * abs(gw["dtheta"])


@pytest.mark.parametrize("W,alpha,full_dtheta", [
    (8, 0.5 + 5 / 15, True),          # linear layer 5: fl64(alpha * 144) just below 120
    (8, 0.5 + (7 * 6 % 16) / 15, True),   # coprime layer 6 (alpha index 10)
    (6, 0.5 + (7 * 3 % 16) / 15, False),  # coprime layer 3
    (10, 0.5 + 11 / 15, False),       # linear layer 11
    (12, 1.5, False),                 # last linear layer
])
def test_config2_bf16_interp(sfa, W, alpha, full_dtheta):
    x = si.make_qkvdo(32, 1024, 8, 2, 64, "bf16", seed=si.mix_seed(0, 2), layer=int(alpha * 100))
    slots = o.interp_slots(FIB, alpha, W)
    fwd = lambda d: sfa.forward(d["q"], d["k"], d["v"], W=W, alpha=alpha, base=FIB)
    bwd = lambda d, O, L: sfa.backward(d["q"], d["k"], d["v"], O, L, d["do"], W=W, alpha=alpha, base=FIB)
    _, _, g = _sampled(sfa, x, [(0, 0), (31, 1), (17, 0)], slots, 1e4, fwd, bwd, True)
    if full_dtheta:
        gw = o.backward(x["q"], x["k"], x["v"], x["do"], slots, 1e4, alpha=alpha)
        da, dt = _np(g[3])
        check_dalpha_dtheta(da, dt, gw, alpha, True)


@pytest.mark.parametrize("alpha", [1.0, 0.5 + 9 / 15])
def test_config3_pow2(sfa, alpha):
    base = o.pow2_offsets(11)
    x = si.make_qkvdo(32, 1024, 8, 2, 64, "bf16", seed=si.mix_seed(0, 3), layer=int(alpha * 100))
    slots = o.interp_slots(base, alpha, 8)
    fwd = lambda d: sfa.forward(d["q"], d["k"], d["v"], W=8, alpha=alpha, base=base)
    bwd = lambda d, O, L: sfa.backward(d["q"], d["k"], d["v"], O, L, d["do"], W=8, alpha=alpha, base=base)
    _sampled(sfa, x, [(5, 1), (30, 0)], slots, 1e4, fwd, bwd, True)


def test_config3_integer_path(sfa):
    """Config 3 at alpha = 1 through the integer path (window 0..8 and the
    powers of two as exact one-row gathers: the rung kernels' integer pairs,
    one tile per pair, and the two-k-step key side); sampled units."""
    dist = sorted(set(range(9)) | set(o.pow2_offsets(11)))
    x = si.make_qkvdo(32, 1024, 8, 2, 64, "bf16", seed=si.mix_seed(0, 33), layer=3)
    fwd = lambda d: sfa.forward_int(d["q"], d["k"], d["v"], dist=dist)
    bwd = lambda d, O, L: sfa.backward_int(d["q"], d["k"], d["v"], O, L, d["do"], dist=dist)
    assert sfa.band_plan(dist, 1024, 4)[0] == 0  # the rung kernels, not the band ones
    _sampled(sfa, x, [(2, 0), (31, 1)], o.dist_slots(dist), 1e4, fwd, bwd, True)


@pytest.mark.parametrize("T,alpha", [(2048, 0.5), (4096, 1.0), (8192, 1.0), (16384, 1.5)])
def test_config4_int_forward_long(sfa, T, alpha):
    dist = o.int_distances(FIB, alpha, 8)
    x = si.make_qkvdo(4, T, 8, 2, 64, "bf16", seed=si.mix_seed(0, 4), layer=T, with_do=False)
    fwd = lambda d: sfa.forward_int(d["q"], d["k"], d["v"], dist=dist)
    _sampled(sfa, x, [(3, 1)], o.dist_slots(dist), 1e4, fwd, None, True, check_bwd=False)


def test_config5_christoffel(sfa):
    dist = o.christoffel_offsets(128, 1024, include_zero=True)
    assert len(dist) == 129 and dist[:3] == [0, 7, 15]
    x = si.make_qkvdo(16, 2048, 4, 4, 64, "bf16", seed=si.mix_seed(0, 5))
    fwd = lambda d: sfa.forward_int(d["q"], d["k"], d["v"], dist=dist)
    bwd = lambda d, O, L: sfa.backward_int(d["q"], d["k"], d["v"], O, L, d["do"], dist=dist)
    _sampled(sfa, x, [(9, 2)], o.dist_slots(dist), 1e4, fwd, bwd, True)


def test_long_sequence_backward(sfa):
    """Interpolated forward and backward at T = 8192 (one sequence; many rung
    slabs far from the tile), checked on one (batch, KV head) unit; dL/dalpha
    over the whole call."""
    alpha = 1.37
    x = si.make_qkvdo(1, 8192, 8, 2, 64, "bf16", seed=si.mix_seed(0, 8), layer=8192)
    slots = o.interp_slots(FIB, alpha, 8)
    fwd = lambda d: sfa.forward(d["q"], d["k"], d["v"], W=8, alpha=alpha, base=FIB)
    bwd = lambda d, O, L: sfa.backward(d["q"], d["k"], d["v"], O, L, d["do"], W=8, alpha=alpha, base=FIB)
    _, _, g = _sampled(sfa, x, [(0, 1)], slots, 1e4, fwd, bwd, True)
    gw = o.backward(x["q"], x["k"], x["v"], x["do"], slots, 1e4, alpha=alpha)
    da, dt = _np(g[3])
    check_dalpha_dtheta(da, dt, gw, alpha, True)
