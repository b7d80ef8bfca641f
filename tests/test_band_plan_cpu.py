"""Host logic of the band layout (sfa_band_plan): the runs it returns are
arithmetic progressions of one step delta dividing T, and together they are
exactly the distances d with |d| < T (negative ones read later keys); the
chosen delta minimises the tile count.  Where the rung kernels could take the
set (G = 4 or 8, no negative distance), sets the band kernels would serve
badly (fewer than 8 distances per tile) get no plan; elsewhere every plan is
used (the alternative is the SIMT path)."""
import itertools
import random

import pytest

import oracle as o


@pytest.fixture(scope="module")
def sfa(sfa_lib):
    import static_offset_sparse_gb300 as s

    return s


def _tiles(runs, G):
    bu = 64 // G
    return sum((bu + n - 1 + 63) // 64 for _, n in runs)


def _brute_best(dist, T, G):
    """Smallest tile count over every step <= 64 dividing T, by brute force."""
    S = sorted(d for d in set(dist) if -T < d < T)
    best = None
    for delta in range(1, 65):
        if T % delta or delta > T:
            continue
        runs, left = [], set(S)
        for d in S:
            if d not in left:
                continue
            n = 0
            while d + n * delta in left:
                left.discard(d + n * delta)
                n += 1
            runs.append((d, n))
        if len(runs) > 128:
            continue
        c = _tiles(runs, G)
        if best is None or c < best[0]:
            best = (c, delta)
    return best


def _rung_ok(dist, G):
    return G in (4, 8) and min(dist) >= 0


def _check_plan(sfa, dist, T, G):
    delta, runs = sfa.band_plan(dist, T, G)
    if delta == 0:
        assert runs == []
        return delta, runs
    assert T % delta == 0 and 1 <= delta <= 64
    covered = []
    for a, n in runs:
        assert n >= 1
        covered += [a + delta * t for t in range(n)]
    assert sorted(covered) == sorted(d for d in set(dist) if -T < d < T)
    assert [a for a, _ in runs] == sorted(a for a, _ in runs)
    # maximal runs: a run's start has no predecessor in the set
    for a, _ in runs:
        assert a - delta not in set(dist)
    return delta, runs


@pytest.mark.parametrize("m,k", [(128, 1024), (32, 256), (16, 64), (64, 512)])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_christoffel_is_one_run(sfa, m, k, G):
    dist = o.christoffel_offsets(m, k, include_zero=True)
    T = 2048
    delta, runs = _check_plan(sfa, dist, T, G)
    want = _brute_best(dist, T, G)
    if delta:
        assert delta == k // m
        assert runs == [(0, 1), (k // m - 1, m)]
        assert _tiles(runs, G) == want[0]
        assert len(set(dist)) >= 8 * want[0] or not _rung_ok(dist, G)
    else:
        assert _rung_ok(dist, G) and len(set(dist)) < 8 * want[0]


def test_config5_plan(sfa):
    dist = o.christoffel_offsets(128, 1024, include_zero=True)
    assert sfa.band_plan(dist, 2048, 1) == (8, [(0, 1), (7, 128)])


@pytest.mark.parametrize("W", [15, 63, 127, 500])
def test_window_is_step_one(sfa, W):
    assert sfa.band_plan(list(range(W + 1)), 1024, 1) == (1, [(0, W + 1)])


def test_full_causal_and_distances_past_T(sfa):
    assert sfa.band_plan(list(range(1000)), 1000, 4) == (1, [(0, 1000)])
    # distances >= T reach no key and are left out
    assert sfa.band_plan(list(range(2000)), 1000, 4) == (1, [(0, 1000)])


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_fibonacci_and_pow2(sfa, G):
    """Singleton rungs: no plan where the rung kernels take the set (G = 4, 8);
    at G = 1, 2 the plan of step 1 (window run + singletons) beats SIMT."""
    fib = sorted(set(range(9)) | set(sfa.offsets_fib(15)))
    pow2 = sorted(set(range(9)) | set(sfa.offsets_pow2(11)))
    for dist in (fib, pow2):
        delta, runs = _check_plan(sfa, dist, 1024, G)
        if G in (4, 8):
            assert (delta, runs) == (0, [])
        else:
            assert delta == 1 and runs[0] == (0, 9)


def test_no_plan_cases(sfa):
    ch = o.christoffel_offsets(128, 1024, include_zero=True)
    assert sfa.band_plan(ch, 2047, 4) == (0, [])            # 8 does not divide T
    assert _check_plan(sfa, ch, 2047, 1)[0] in (1, 23)       # G = 1: another step
    assert sfa.band_plan(ch, 2048, 16) == (0, [])           # G outside 1, 2, 4, 8
    assert sfa.band_plan(ch, 2048, 3) == (0, [])
    assert sfa.band_plan(ch[1:], 2048, 1) == (0, [])        # no distance 0


def test_signed_sets_are_runs(sfa):
    """Bidirectional sets: the Christoffel offsets and their negatives are
    three runs of step k / m; distances with |d| >= T are left out."""
    ch = o.signed_christoffel_offsets(128, 1024)
    assert sfa.band_plan(ch, 2048, 1) == (8, [(-1023, 128), (0, 1), (7, 128)])
    assert sfa.band_plan(ch, 512, 1) == (8, [(-511, 64), (0, 1), (7, 64)])
    assert sfa.band_plan(list(range(-40, 41)), 1024, 4) == (1, [(-40, 81)])
    assert sfa.band_plan([-3] + o.christoffel_offsets(128, 1024, True), 2048, 1) == \
        (8, [(-3, 1), (0, 1), (7, 128)])
    for G in (1, 2, 4, 8):
        _check_plan(sfa, ch, 2048, G)


def test_capacity(sfa):
    import ctypes as C

    from static_offset_sparse_gb300 import _lib

    arr, n = _lib.i32_array(list(range(16)) + [19 + 4 * t for t in range(80)])
    d, nr = C.c_int32(0), C.c_int32(0)
    starts = (C.c_int32 * 2)()
    lens = (C.c_int32 * 2)()
    rc = _lib._lib().sfa_band_plan(arr, n, 1024, 4, C.byref(d), starts, lens, 2, C.byref(nr))
    assert rc == 3 and d.value == 4 and nr.value == 4  # SFA_ERR_CAPACITY, counts still set


def test_random_sets_match_brute_force(sfa):
    rng = random.Random(7)
    for _ in range(60):
        T = rng.choice([256, 512, 600, 1024])
        G = rng.choice([1, 2, 4, 8])
        step = rng.choice([1, 2, 3, 4, 8])
        dist = {0}
        signed = rng.random() < 0.4
        for _ in range(rng.randint(1, 4)):
            a = rng.randrange(-T if signed else 0, T)
            n = rng.randint(1, 200)
            dist |= {a + step * t for t in range(n)}
        dist |= set(rng.sample(range(-T if signed else 0, T), rng.randint(0, 5)))
        dist = sorted(dist)
        delta, runs = _check_plan(sfa, dist, T, G)
        best = _brute_best(dist, T, G)
        m = len([d for d in dist if -T < d < T])
        if delta:
            assert _tiles(runs, G) == best[0] and delta == best[1]
        elif _rung_ok(dist, G):
            assert best is None or m < 8 * best[0]
        else:
            assert best is None


def test_plan_is_order_and_duplicate_free(sfa):
    ch = o.christoffel_offsets(32, 256, include_zero=True)
    shuffled = list(itertools.chain(ch[::-1], ch[:5]))
    assert sfa.band_plan(shuffled, 1024, 1) == sfa.band_plan(ch, 1024, 1)
