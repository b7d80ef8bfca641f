"""Bounds shared by the GPU parity tests."""
import numpy as np

# max-abs bound on O, dQ, dK, dV for bf16 and fp32 I/O
BF16_TOL = 2e-2
F32_TOL = 1e-5


def bf16_half_ulp(x):
    """Half a unit in the last place of bf16 at each |x|.

    bf16 keeps 8 significant bits, so for 2^e <= |x| < 2^(e+1) neighbouring
    values are 2^(e-7) apart and round-to-nearest moves a value by at most
    2^(e-8).  Below the smallest normal (2^-126) the spacing is 2^-133.
    Zero rounds to itself.
    """
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(np.maximum(e, -126.0) - 8.0), 0.0)


def bf16_bound(want, tol=BF16_TOL):
    """Per-element bound for a bf16 output: the flat max-abs tol plus the
    output's own rounding, half a bf16 ulp of the exact value.  A bf16 number
    cannot land closer to the exact value than that rounding: for |x| >= 8
    half an ulp (2^-5 and up) alone exceeds 2e-2."""
    return tol + bf16_half_ulp(want)


def check_close(name, got, want, bf16, tol=None, report=True):
    """Element-by-element check of got against the oracle's want.

    fp32: |got - want| <= tol (1e-5).  bf16: |got - want| <= tol (2e-2) plus
    half a bf16 ulp of want, i.e. every element above the flat tol is above
    it by no more than its own output rounding.  Prints the max-abs error and
    the count of elements above the flat tol.
    """
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, f"{name}: shape {got.shape} != {want.shape}"
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    if not want.size:
        return 0.0
    tol = tol if tol is not None else (BF16_TOL if bf16 else F32_TOL)
    err = np.abs(got - want)
    lim = bf16_bound(want, tol) if bf16 else tol
    excess = err - lim
    worst = np.unravel_index(np.argmax(excess), excess.shape)
    over = int((err > tol).sum())
    if report:
        print(f"{name}: max-abs {err.max():.3g}; {over} of {err.size} above {tol:g}"
              + (f" (each within half a bf16 ulp of the exact value)" if bf16 and over and excess[worst] <= 0 else ""))
    assert excess[worst] <= 0, (
        f"{name}: |err| {err[worst]:.3g} at {worst} (exact {want[worst]:.4g}) > bound "
        f"{lim if np.isscalar(lim) else lim[worst]:.3g}")
    return float(err.max())


def dalpha_tol(gw, bf16):
    """Bound on |dL/dalpha - exact|.

    fp32 I/O: 1e-3 relative.  bf16 I/O (no bound on the pages for bf16): the
    (position, dimension) terms of dL/dalpha are products of bf16-rounded
    operands and cancel (their absolute sum can exceed |dL/dalpha| by 10^3),
    so the rounding error grows like a random walk over them: 2e-2 relative
    plus 2^-6 (4 bf16 units) times the root-sum-square of the terms, the
    oracle's dalpha_rss.  The observed errors of the small cases stay within
    about half of that second part; a wrong or dropped term misses by the
    terms' absolute sum, two orders of magnitude more.
    """
    if not bf16:
        return 1e-3 * abs(gw["dalpha"])
    return 2e-2 * abs(gw["dalpha"]) + 2.0 ** -6 * gw["dalpha_rss"]


def check_dalpha_dtheta(da, dt, gw, alpha, bf16):
    tol = dalpha_tol(gw, bf16)
    assert abs(da - gw["dalpha"]) <= tol + 1e-9, (da, gw["dalpha"], tol)
    scale = abs((alpha - 0.5) * (1.5 - alpha))  # dtheta = dalpha (alpha - 1/2)(3/2 - alpha)
    assert abs(dt - gw["dtheta"]) <= tol * scale + 1e-9, (dt, gw["dtheta"], tol * scale)
