"""GPU parity of the band kernels: integer bf16 distance sets that split into
long arithmetic runs of one step delta (the Christoffel carry-word offsets
of "Christoffel-Balanced Sparse Attention" with m | k, dense windows, the
full causal set, and mixed windows with a strided tail), for G = 1, 2, 4
and 8 query heads per KV head.  Forward and backward against the fp64
oracle on the same seeded inputs, with the bounds of the other parity
tests; ragged tails (T / delta not a multiple of the tile) included."""
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


def _check(name, got, want):
    check_close(name, got, want, True)


SETS = {
    "christoffel32_256": o.christoffel_offsets(32, 256, include_zero=True),
    "christoffel128_1024": o.christoffel_offsets(128, 1024, include_zero=True),
    "window64": list(range(64)),
    "window_stride4": list(range(16)) + [19 + 4 * t for t in range(80)],
}
# (B, T, Hq, Hkv): G = 1, 2, 4, 8; T / delta leaves a ragged last tile
SHAPES = [(1, 200, 2, 2), (2, 456, 4, 2), (1, 1000, 8, 2), (1, 456, 8, 1)]
CASES = [(n, s) for n in sorted(SETS) for s in SHAPES
         if not (n == "window_stride4" and s[1] == 200)]


def _run(sfa, x, dist, theta, k_rot=False):
    import torch

    dev = {n: t.cuda() for n, t in x.items()}
    kw = {}
    if k_rot:
        kw["k_rot"] = sfa.rope_keys(dev["k"], rope_theta=theta)
    O, L = sfa.forward_int(dev["q"], dev["k"], dev["v"], dist=dist, rope_theta=theta, **kw)
    g = sfa.backward_int(dev["q"], dev["k"], dev["v"], O, L, dev["do"], dist=dist,
                         rope_theta=theta, **kw)
    torch.cuda.synchronize()
    assert sfa.get_device_status() == 0
    return O, L, g


def _f64(t):
    import torch

    return t.detach().to("cpu", torch.float64).numpy()


@pytest.mark.parametrize("name,shape", CASES)
def test_band_forward_backward(sfa, name, shape):
    B, T, Hq, Hkv = shape
    dist = SETS[name]
    delta, runs = sfa.band_plan(dist, T, Hq // Hkv)
    assert delta > 0, "the set must take the band kernels"
    x = si.make_qkvdo(B, T, Hq, Hkv, 64, "bf16", seed=1300 + T + len(dist))
    O, L, (dq, dk, dv) = _run(sfa, x, dist, 1e4)
    slots = o.dist_slots(dist)
    Ow, Lw = o.forward(x["q"], x["k"], x["v"], slots, 1e4)
    gw = o.backward(x["q"], x["k"], x["v"], x["do"], slots, 1e4)
    _check("O", _f64(O), Ow)
    assert np.abs(_f64(L) - Lw).max() <= 2e-2
    _check("dQ", _f64(dq), gw["dq"])
    _check("dK", _f64(dk), gw["dk"])
    _check("dV", _f64(dv), gw["dv"])


@pytest.mark.parametrize("shape", SHAPES)
def test_band_full_causal(sfa, shape):
    """Every distance 0..T-1: dense causal attention as one run of step 1."""
    B, T, Hq, Hkv = shape
    dist = list(range(T))
    assert sfa.band_plan(dist, T, Hq // Hkv) == (1, [(0, T)])
    x = si.make_qkvdo(B, T, Hq, Hkv, 64, "bf16", seed=1400 + T)
    O, L, (dq, dk, dv) = _run(sfa, x, dist, 1e4)
    slots = o.dist_slots(dist)
    Ow, Lw = o.forward(x["q"], x["k"], x["v"], slots, 1e4)
    gw = o.backward(x["q"], x["k"], x["v"], x["do"], slots, 1e4)
    _check("O", _f64(O), Ow)
    assert np.abs(_f64(L) - Lw).max() <= 2e-2
    _check("dQ", _f64(dq), gw["dq"])
    _check("dK", _f64(dk), gw["dk"])
    _check("dV", _f64(dv), gw["dv"])


@pytest.mark.parametrize("G", [1, 4])
def test_band_no_rope(sfa, G):
    dist = SETS["christoffel32_256"]
    B, T, Hkv = 1, 512, 2
    x = si.make_qkvdo(B, T, G * Hkv, Hkv, 64, "bf16", seed=1500 + G)
    O, L, (dq, dk, dv) = _run(sfa, x, dist, 0.0)
    slots = o.dist_slots(dist)
    Ow, Lw = o.forward(x["q"], x["k"], x["v"], slots, 0.0)
    gw = o.backward(x["q"], x["k"], x["v"], x["do"], slots, 0.0)
    _check("O", _f64(O), Ow)
    _check("dQ", _f64(dq), gw["dq"])
    _check("dK", _f64(dk), gw["dk"])
    _check("dV", _f64(dv), gw["dv"])


def test_band_k_rot_reuse_is_bit_identical(sfa):
    """Rotated keys handed in (one rotation shared by forward and backward)
    give the same bits as rotating inside each call."""
    import torch

    dist = SETS["christoffel128_1024"]
    x = si.make_qkvdo(2, 1024, 4, 4, 64, "bf16", seed=1600)
    a = _run(sfa, x, dist, 1e4)
    b = _run(sfa, x, dist, 1e4, k_rot=True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    for u, w in zip(a[2], b[2]):
        assert torch.equal(u, w)


def test_band_is_deterministic(sfa):
    import torch

    dist = SETS["window_stride4"]
    x = si.make_qkvdo(1, 1000, 8, 2, 64, "bf16", seed=1700)
    a = _run(sfa, x, dist, 1e4)
    b = _run(sfa, x, dist, 1e4)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    for u, w in zip(a[2], b[2]):
        assert torch.equal(u, w)


@pytest.mark.parametrize("G", [1, 4])
def test_band_fallback_when_delta_does_not_divide_T(sfa, G):
    """T = 201 is not a multiple of the Christoffel step 8.  G = 4: no band
    plan, the set runs the rung kernels; G = 1: the plan of step 1 (every
    distance its own run, still ahead of the SIMT path).  Same result."""
    dist = SETS["christoffel32_256"]
    B, T, Hkv = 1, 201, 2
    assert sfa.band_plan(dist, T, G)[0] == (0 if G == 4 else 1)
    x = si.make_qkvdo(B, T, G * Hkv, Hkv, 64, "bf16", seed=1800 + G)
    O, L, (dq, dk, dv) = _run(sfa, x, dist, 1e4)
    slots = o.dist_slots(dist)
    Ow, _ = o.forward(x["q"], x["k"], x["v"], slots, 1e4)
    gw = o.backward(x["q"], x["k"], x["v"], x["do"], slots, 1e4)
    _check("O", _f64(O), Ow)
    _check("dQ", _f64(dq), gw["dq"])
    _check("dK", _f64(dk), gw["dk"])
    _check("dV", _f64(dv), gw["dv"])


def test_band_christoffel_gqa_full_size_sampled(sfa):
    """The Christoffel 128/1024 set with 8 query heads over 2 KV heads (G = 4,
    formerly the rung kernels) at B = 4, T = 2048; one (batch, KV head) unit
    against the oracle."""
    import torch

    dist = SETS["christoffel128_1024"]
    x = si.make_qkvdo(4, 2048, 8, 2, 64, "bf16", seed=1900)
    O, L, (dq, dk, dv) = _run(sfa, x, dist, 1e4)
    rows = [(3, 1)]
    slots = o.dist_slots(dist)
    Ow, Lw = o.forward(x["q"], x["k"], x["v"], slots, 1e4, rows=rows)
    gw = o.backward(x["q"], x["k"], x["v"], x["do"], slots, 1e4, rows=rows)
    b, g = rows[0]
    hs = slice(4 * g, 4 * g + 4)
    _check("O", _f64(O)[b, hs], Ow[b, hs])
    assert np.abs(_f64(L)[b, hs] - Lw[b, hs]).max() <= 2e-2
    _check("dQ", _f64(dq)[b, hs], gw["dq"][b, hs])
    _check("dK", _f64(dk)[b, g], gw["dk"][b, g])
    _check("dV", _f64(dv)[b, g], gw["dv"][b, g])
    assert torch.isfinite(dk).all() and torch.isfinite(dv).all()


@pytest.mark.parametrize("T,Hq,Hkv", [(16, 2, 2), (16, 8, 1), (65, 4, 4), (65, 8, 2), (130, 4, 2)])
def test_band_tiny_and_ragged(sfa, T, Hq, Hkv):
    """Whole sequence in one partial tile (T = 16), one row past a tile (T = 65),
    full causal sets; results against the oracle."""
    dist = list(range(T))
    delta, runs = sfa.band_plan(dist, T, Hq // Hkv)
    assert delta == 1 and runs == [(0, T)]
    x = si.make_qkvdo(2, T, Hq, Hkv, 64, "bf16", seed=2000 + T + Hq)
    O, L, (dq, dk, dv) = _run(sfa, x, dist, 1e4)
    slots = o.dist_slots(dist)
    Ow, Lw = o.forward(x["q"], x["k"], x["v"], slots, 1e4)
    gw = o.backward(x["q"], x["k"], x["v"], x["do"], slots, 1e4)
    _check("O", _f64(O), Ow)
    assert np.abs(_f64(L) - Lw).max() <= 2e-2
    _check("dQ", _f64(dq), gw["dq"])
    _check("dK", _f64(dk), gw["dk"])
    _check("dV", _f64(dv), gw["dv"])


def test_band_distances_past_T_are_ignored(sfa):
    """Distances >= T reach no key: the set with them gives the same bits as
    the set without them."""
    import torch

    ch = SETS["christoffel32_256"]
    T = 192
    assert sfa.band_plan(ch, T, 1) == (8, [(0, 1), (7, 24)])
    x = si.make_qkvdo(1, T, 4, 4, 64, "bf16", seed=2100)
    a = _run(sfa, x, [d for d in ch if d < T], 1e4)
    b = _run(sfa, x, ch, 1e4)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    for u, w in zip(a[2], b[2]):
        assert torch.equal(u, w)


def _random_band_cases(n, seed):
    """Seeded run-structured sets that get a band plan with step >= 2 and at
    least two runs: steps 2, 3, 4, 5, 8, runs starting past the step (several
    runs in one key class), distances past T, ragged T / delta."""
    import random

    import static_offset_sparse_gb300 as s

    rng = random.Random(seed)
    out = []
    while len(out) < n:
        delta = rng.choice([2, 3, 4, 5, 8])
        G = rng.choice([1, 2, 4, 8])
        T = delta * rng.randint(20, 90)
        dist = {0}
        for _ in range(rng.randint(1, 3)):
            a = rng.randrange(0, 3 * delta + 5)
            dist |= {a + delta * t for t in range(rng.randint(20, 120))}
        dist = sorted(dist)
        d, runs = s.band_plan(dist, T, G)
        if d >= 2 and len(runs) >= 2:
            out.append((T, G, dist))
    return out


@pytest.mark.parametrize("case", range(12))
def test_band_random_run_sets(sfa, case):
    T, G, dist = _random_band_cases(12, 11)[case]
    Hkv = 2 if G <= 4 else 1
    x = si.make_qkvdo(1, T, G * Hkv, Hkv, 64, "bf16", seed=2200 + case)
    O, L, (dq, dk, dv) = _run(sfa, x, dist, 1e4)
    slots = o.dist_slots(dist)
    Ow, Lw = o.forward(x["q"], x["k"], x["v"], slots, 1e4)
    gw = o.backward(x["q"], x["k"], x["v"], x["do"], slots, 1e4)
    _check("O", _f64(O), Ow)
    assert np.abs(_f64(L) - Lw).max() <= 2e-2
    _check("dQ", _f64(dq), gw["dq"])
    _check("dK", _f64(dk), gw["dk"])
    _check("dV", _f64(dv), gw["dv"])


@pytest.mark.parametrize("name,shape", [("christoffel32_256", (1, 200, 2, 2)),
                                        ("christoffel128_1024", (2, 2048, 4, 4)),
                                        ("window64", (2, 456, 4, 2)),
                                        ("window_stride4", (1, 1000, 8, 2)),
                                        ("christoffel32_256", (1, 456, 8, 1))])
def test_band_forward_both_kernels(sfa, sfa_lib, name, shape):
    """The band forward on the fifth-generation tensor cores (tcgen05, TMEM
    accumulators, 128 query rows per CTA) and on mma.sync (64 rows per CTA):
    each against the oracle, and against each other."""
    import torch

    B, T, Hq, Hkv = shape
    dist = SETS[name]
    x = si.make_qkvdo(B, T, Hq, Hkv, 64, "bf16", seed=1700 + T + len(dist))
    dev = {n: t.cuda() for n, t in x.items()}
    Ow, Lw = o.forward(x["q"], x["k"], x["v"], o.dist_slots(dist), 1e4)
    outs = {}
    try:
        for opt in (1, 0):
            assert sfa_lib.sfa_set_option(0, opt) == 0
            O, L = sfa.forward_int(dev["q"], dev["k"], dev["v"], dist=dist)
            torch.cuda.synchronize()
            assert sfa.get_device_status() == 0
            _check(f"O (tcgen05={opt})", _f64(O), Ow)
            assert np.abs(_f64(L) - Lw).max() <= 2e-2
            outs[opt] = (_f64(O), _f64(L))
    finally:
        assert sfa_lib.sfa_set_option(0, 0) == 0  # the default
    assert np.abs(outs[0][1] - outs[1][1]).max() <= 1e-4  # LSE: same keys, fp32 logits
    assert np.abs(outs[0][0] - outs[1][0]).max() <= 2e-2
