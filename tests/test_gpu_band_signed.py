"""GPU parity of the band kernels on signed (bidirectional) distance sets:
"Christoffel-Balanced Sparse Attention" allows signed offsets for
bidirectional attention, a negative distance s reading the later key
i + |s|.  Such sets split into runs like causal ones (the Christoffel offsets
and their negatives are three runs of step k / m); the band walks clip every
band to the sequence at both ends.  Forward and backward against the fp64
oracle, G = 1, 2, 4 and 8, ragged tails, the fully bidirectional set (dense
non-causal attention as one run of step 1), seeded random signed run sets,
and the signed Christoffel 128/1024 set at the benchmark's size (sampled)."""
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


def _f64(t):
    import torch

    return t.detach().to("cpu", torch.float64).numpy()


def _run(sfa, x, dist, theta=1e4):
    import torch

    dev = {n: t.cuda() for n, t in x.items()}
    O, L = sfa.forward_int(dev["q"], dev["k"], dev["v"], dist=dist, rope_theta=theta)
    g = sfa.backward_int(dev["q"], dev["k"], dev["v"], O, L, dev["do"], dist=dist, rope_theta=theta)
    torch.cuda.synchronize()
    assert sfa.get_device_status() == 0
    return O, L, g


def _compare(x, O, L, g, dist, theta=1e4, rows=None):
    slots = o.dist_slots(dist)
    Ow, Lw = o.forward(x["q"], x["k"], x["v"], slots, theta, rows=rows)
    gw = o.backward(x["q"], x["k"], x["v"], x["do"], slots, theta, rows=rows)
    dq, dk, dv = g
    if rows is None:
        check_close("O", _f64(O), Ow, True)
        assert np.abs(_f64(L) - Lw).max() <= 2e-2
        check_close("dQ", _f64(dq), gw["dq"], True)
        check_close("dK", _f64(dk), gw["dk"], True)
        check_close("dV", _f64(dv), gw["dv"], True)
        return
    G = x["q"].shape[1] // x["k"].shape[1]
    for b, g_ in rows:
        hs = slice(G * g_, G * g_ + G)
        check_close("O", _f64(O)[b, hs], Ow[b, hs], True)
        assert np.abs(_f64(L)[b, hs] - Lw[b, hs]).max() <= 2e-2
        check_close("dQ", _f64(dq)[b, hs], gw["dq"][b, hs], True)
        check_close("dK", _f64(dk)[b, g_], gw["dk"][b, g_], True)
        check_close("dV", _f64(dv)[b, g_], gw["dv"][b, g_], True)


SETS = {
    "signed_christoffel32_256": o.signed_christoffel_offsets(32, 256),
    "signed_window40": list(range(-40, 41)),
    "window_and_later_stride4": list(range(9)) + [-3 - 4 * t for t in range(50)],
}
SHAPES = [(1, 200, 2, 2), (2, 456, 4, 2), (1, 1000, 8, 2), (1, 456, 8, 1)]


CASES = [(n, s) for n in sorted(SETS) for s in SHAPES
         if not (n == "window_and_later_stride4" and s[1] == 200)]  # no plan there


@pytest.mark.parametrize("name,shape", CASES)
def test_signed_band_forward_backward(sfa, name, shape):
    B, T, Hq, Hkv = shape
    dist = SETS[name]
    delta, runs = sfa.band_plan(dist, T, Hq // Hkv)
    assert delta > 0 and runs[0][0] < 0, "the set must take the band kernels"
    x = si.make_qkvdo(B, T, Hq, Hkv, 64, "bf16", seed=3100 + T + len(dist))
    O, L, g = _run(sfa, x, dist)
    _compare(x, O, L, g, dist)


@pytest.mark.parametrize("T,Hq,Hkv", [(16, 2, 2), (65, 4, 4), (130, 8, 2), (200, 8, 1)])
def test_fully_bidirectional_is_dense_attention(sfa, T, Hq, Hkv):
    """Every distance -(T-1) .. T-1: plain (non-causal) softmax attention, one
    run of step 1; the oracle's masked softmax over all keys."""
    dist = list(range(-(T - 1), T))
    assert sfa.band_plan(dist, T, Hq // Hkv) == (1, [(-(T - 1), 2 * T - 1)])
    x = si.make_qkvdo(2, T, Hq, Hkv, 64, "bf16", seed=3200 + T)
    O, L, g = _run(sfa, x, dist)
    _compare(x, O, L, g, dist)


def _random_signed_cases(n, seed):
    """Seeded signed run sets with a band plan of step >= 2: runs starting at
    negative and positive distances, distances past the sequence either way,
    ragged T / delta."""
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
            a = rng.randrange(-T - 10, 3 * delta + 5)
            dist |= {a + delta * t for t in range(rng.randint(20, 120))}
        dist = sorted(dist)
        d, runs = s.band_plan(dist, T, G)
        if d >= 2 and len(runs) >= 2 and runs[0][0] < 0:
            out.append((T, G, dist))
    return out


@pytest.mark.parametrize("case", range(10))
def test_signed_band_random_run_sets(sfa, case):
    T, G, dist = _random_signed_cases(10, 23)[case]
    Hkv = 2 if G <= 4 else 1
    x = si.make_qkvdo(1, T, G * Hkv, Hkv, 64, "bf16", seed=3300 + case)
    O, L, g = _run(sfa, x, dist)
    _compare(x, O, L, g, dist)


def test_signed_christoffel_full_size_sampled(sfa):
    """The signed Christoffel 128/1024 set at B = 16, T = 2048, 4/4 heads (the
    bench's bidirectional line): two (batch, KV head) units against the
    oracle, the rest finite."""
    import torch

    dist = o.signed_christoffel_offsets(128, 1024)
    assert sfa.band_plan(dist, 2048, 1)[0] == 8
    x = si.make_qkvdo(16, 2048, 4, 4, 64, "bf16", seed=3400)
    O, L, g = _run(sfa, x, dist)
    _compare(x, O, L, g, dist, rows=[(0, 0), (15, 3)])
    for t in (O, *g):
        assert torch.isfinite(t).all()


def test_signed_band_forward_both_kernels(sfa, sfa_lib):
    """The tcgen05 band forward and the mma.sync one on a signed set."""
    import torch

    dist = SETS["signed_christoffel32_256"]
    x = si.make_qkvdo(2, 456, 4, 2, 64, "bf16", seed=3500)
    dev = {n: t.cuda() for n, t in x.items()}
    Ow, Lw = o.forward(x["q"], x["k"], x["v"], o.dist_slots(dist), 1e4)
    try:
        for opt in (1, 0):
            assert sfa_lib.sfa_set_option(0, opt) == 0
            O, L = sfa.forward_int(dev["q"], dev["k"], dev["v"], dist=dist)
            torch.cuda.synchronize()
            assert sfa.get_device_status() == 0
            check_close(f"O (tcgen05={opt})", _f64(O), Ow, True)
            assert np.abs(_f64(L) - Lw).max() <= 2e-2
    finally:
        assert sfa_lib.sfa_set_option(0, 0) == 0


def test_signed_long_sequence_sampled(sfa):
    """T = 8192 (128 key tiles per class at step 8): the signed Christoffel
    128/1024 set, one (batch, KV head) unit against the oracle, G = 4."""
    import torch

    dist = o.signed_christoffel_offsets(128, 1024)
    x = si.make_qkvdo(1, 8192, 8, 2, 64, "bf16", seed=3600)
    O, L, g = _run(sfa, x, dist)
    _compare(x, O, L, g, dist, rows=[(0, 1)])
    for t in (O, *g):
        assert torch.isfinite(t).all()
