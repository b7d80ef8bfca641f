"""Bounds shared by the GPU parity tests."""


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
