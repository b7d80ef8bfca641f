"""CPU tests of the offset-schedule analysis and the shared power-law list
(host code in libsfa) against the oracle's independent definitions: integer
results bit for bit."""
import numpy as np
import pytest

import oracle as o
import sfa_inputs as si

FIB = o.fib_offsets(15)


@pytest.fixture(scope="module")
def s(sfa_lib):
    import static_offset_sparse_gb300 as m

    return m


def _random_sets(seed, L, T, nmax):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(L):
        n = int(rng.integers(1, nmax + 1))
        S = rng.integers(0, T + 5, size=n).tolist()  # duplicates and d >= T included
        if rng.random() < 0.7:
            S.append(0)
        out.append(S)
    return out


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 129, 1000])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_reach_random_sets(s, T, seed):
    sets = _random_sets(seed * 1000 + T, 1 + seed * 3, T, 6)
    _same(s.reach(sets, T), o.reach(sets, T))


def _same(a, b):
    assert list(a[0]) == list(b[0]) and list(a[1]) == list(b[1])


def test_reach_staggered_fibonacci_stack(s):
    """The 16-layer integer stack (alpha_l linear, rounded; W = 8)."""
    T = 4096
    sets = [o.int_distances(FIB, 0.5 + l / 15, 8) for l in range(16)]
    _same(s.reach(sets, T), o.reach(sets, T))


@pytest.mark.parametrize("m,k,L", [(128, 1024, 8), (64, 512, 3), (3, 8, 5)])
def test_reach_christoffel_stack(s, m, k, L):
    T = 2 * k
    S = o.christoffel_offsets(m, k, include_zero=True)
    hops, cov = s.reach([S] * L, T)
    wh, wc = o.reach([S] * L, T)
    assert hops == wh and cov == wc
    assert s.residue_classes(hops, 8) == o.residue_classes(wh, 8)


def test_histogram(s):
    for dist, T, nb in [(FIB, 1024, 12), ([0, 0, 5, 4096, 7], 1024, 4), (list(range(300)), 256, 10)]:
        assert s.offset_histogram(dist, T, nb) == o.offset_histogram(dist, T, nb)


@pytest.mark.parametrize("sigma", [0.0, 0.5, 0.8, 0.85, 1.2])
@pytest.mark.parametrize("n", [2, 3, 1024, 2048, 100000])
def test_powerlaw_bit_exact(s, sigma, n):
    u = si.uniform(si.mix_seed(21, n, int(sigma * 100)), 64)
    assert s.offsets_powerlaw(u, sigma, n) == o.powerlaw_offsets(u, sigma, n)


def test_errors(s):
    from static_offset_sparse_gb300 import SfaError

    with pytest.raises(SfaError):
        s.reach([[-1, 0]], 10)  # negative distance
    with pytest.raises(SfaError):
        s.offsets_powerlaw([1.0], 0.8, 100)  # u outside [0, 1)
    with pytest.raises(SfaError):
        s.offsets_powerlaw([0.5], -0.1, 100)  # sigma < 0
    with pytest.raises(SfaError):
        s.residue_classes([0, 1, -1], 4)  # M > T
