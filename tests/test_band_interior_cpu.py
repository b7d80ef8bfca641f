"""The band key side's interior test (csrc/sfa_band.cu, band_bwd_kv_kernel).

A 32-query half of a key tile is taken without the per-element test when a
warp-uniform condition on the half's query span and the warp's 16 keys holds.
That is only sound if the condition implies the per-element rule for every
(key row, query column) pair of the warp and the half; this checks the
implication by brute force over random tile geometries (both written out
here as the kernel states them), including rows and columns past the
sequence, negative query starts, every G and both halves.
"""
import random

kBR = 64  # rows of a band tile


def _element_valid(kv, u, Uc, e, length):
    # the kernel's rule: query u reaches key kv through the run iff
    # 0 <= u - kv + e < len, with rows or columns past the sequence excluded
    tb = e - kv if kv < Uc else -(1 << 30)
    uq = u if u < Uc else -(1 << 30)
    return 0 <= uq + tb < length


def _half_full(G, Uc, e, length, vmin, us, hq):
    BU = kBR // G
    ua = us + ((32 * hq) % BU if BU >= 32 else 0)
    ub = ua + min(BU, 32) - 1
    return vmin + 15 < Uc and ub < Uc and ua - (vmin + 15) + e >= 0 and ub - vmin + e <= length - 1


def test_interior_condition_implies_every_element():
    rng = random.Random(7)
    n_full = 0
    for _ in range(40000):
        G = rng.choice([1, 2, 4, 8])
        BU = kBR // G
        Uc = rng.randint(1, 300)
        length = rng.randint(1, 200)
        e = rng.randint(-300, 300)
        v0 = 64 * rng.randint(0, (Uc - 1) // 64)
        us = rng.randint(-100, Uc + 50)
        warp, hq = rng.randint(0, 3), rng.randint(0, 1)
        vmin = v0 + 16 * warp
        if not _half_full(G, Uc, e, length, vmin, us, hq):
            continue
        n_full += 1
        for r in range(16):
            for n in range(32 * hq, 32 * hq + 32):
                assert _element_valid(vmin + r, us + n % BU, Uc, e, length), (G, Uc, length, e, v0, us, warp, hq)
    assert n_full > 500  # the condition is met often enough for the check to mean something


def test_interior_condition_is_met_inside_a_long_run():
    # config 5's long run (len 128) at G = 1: a key tile in the middle of the
    # sequence has halves whose 32 queries all read all 16 keys of a warp
    Uc, length = 256, 128
    hits = 0
    for v0 in (64, 128):
        for warp in range(4):
            vmin = v0 + 16 * warp
            for us in range(0, Uc - 63):
                for hq in range(2):
                    hits += _half_full(1, Uc, 0, length, vmin, us, hq)
    assert hits > 0
