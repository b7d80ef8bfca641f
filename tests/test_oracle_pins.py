"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these re-types the oracle's own formula: each checks a printed value,
a hand-worked example, a closed form, an invariant, a textbook special case,
an independent formulation, or finite differences.
"""
import math
import os

import numpy as np
import pytest

import oracle as o
import sfa_inputs as si

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(x) for x in line.split()])
    return rows


# ---------------------------------------------------------------- offsets


def test_fib_matches_printed_list():
    assert o.fib_offsets(15) == _golden_rows("fib_base.txt")[0]


def test_fib_recurrence_and_reach():
    f = o.fib_offsets(15)
    assert f[0] == 1 and f[1] == 2
    # 987 is the largest Fibonacci number below 1024 (the page's reach remark)
    assert f[-1] < 1024 < f[-1] + f[-2]
    assert all(f[i] == f[i - 1] + f[i - 2] for i in range(2, 15))


def test_pow2_closed_form():
    p = o.pow2_offsets(11)
    assert p == [int(2 ** j) for j in range(11)]
    assert p[-1] == 1024


def test_christoffel_hand_worked_example():
    word, offs = _golden_rows("christoffel_3_8.txt")
    assert o.christoffel_word(3, 8) == word
    assert o.christoffel_offsets(3, 8, include_zero=False) == offs
    assert o.christoffel_offsets(3, 8, include_zero=True) == [0] + offs


@pytest.mark.parametrize("m,k", [(3, 8), (5, 13), (7, 12), (64, 512), (128, 1024), (1, 1), (13, 13), (1, 7)])
def test_christoffel_counts_and_prefix_balance(m, k):
    c = o.christoffel_word(m, k)
    assert len(c) == k and set(c) <= {0, 1}
    assert sum(c) == m  # exactly m ones per period
    pref = np.concatenate([[0], np.cumsum(c)])
    for j in range(k + 1):
        assert abs(pref[j] - j * m / k) < 1.0  # prefix within 1 of j m / k


@pytest.mark.parametrize("m,k", [(3, 8), (5, 13), (7, 12), (4, 10)])
def test_christoffel_balanced_factors(m, k):
    """Sturmian balance: equal-length factors (cyclic) differ by <= 1 one."""
    c = o.christoffel_word(m, k) * 2
    for n in range(1, k + 1):
        counts = {sum(c[s : s + n]) for s in range(k)}
        assert max(counts) - min(counts) <= 1


@pytest.mark.parametrize("m,k", [(64, 512), (128, 1024), (2, 8)])
def test_christoffel_divisible_closed_form(m, k):
    """For m | k the ones sit at j = (k/m)(t+1) - 1: a stride-(k/m) dilation."""
    r = k // m
    assert o.christoffel_offsets(m, k, include_zero=False) == [r * (t + 1) - 1 for t in range(m)]


# ---------------------------------------------------------------- schedules


def test_schedules():
    lin = o.alpha_schedule(16, o.SCHED_LINEAR)
    assert lin[0] == 0.5 and lin[15] == 1.5
    assert all(abs(lin[l] - (0.5 + l / 15)) < 1e-15 for l in range(16))
    assert o.alpha_schedule(16, o.SCHED_FIXED) == [1.0] * 16
    cop = o.alpha_schedule(16, o.SCHED_COPRIME, 7)
    order = _golden_rows("coprime_order_7_16.txt")[0]
    assert sorted(order) == list(range(16))  # a permutation
    assert [order[order[l]] for l in range(16)] == list(range(16))  # involution (49 = 1 mod 16)
    assert cop == [lin[j] for j in order]
    assert sorted(cop) == sorted(lin)  # same multiset
    with pytest.raises(ValueError):
        o.alpha_schedule(16, o.SCHED_COPRIME, 4)


def test_alpha_theta_map():
    assert o.alpha_of_theta(0.0) == 1.0  # learned variant starts at alpha = 1
    for th in (-3.0, -0.2, 0.7, 2.5):
        a = o.alpha_of_theta(th)
        assert 0.5 < a < 1.5
        assert abs(o.theta_of_alpha(a) - th) < 1e-12
    assert o.theta_of_alpha(0.5) == -math.inf and o.theta_of_alpha(1.5) == math.inf


def test_int_distances_rounding():
    want = _golden_rows("int_dist_alpha05.txt")[0]
    got = o.int_distances(o.fib_offsets(), 0.5, -1)  # W = -1: rungs only
    assert got == sorted(set(want))
    # union with the window drops duplicates, keeps 0..W
    d = o.int_distances(o.fib_offsets(), 1.0, 8)
    assert d == list(range(9)) + [13, 21, 34, 55, 89, 144, 233, 377, 610, 987]


def test_interp_rungs_filter_and_weights():
    r = o.interp_rungs(o.fib_offsets(), 1.0, 8)
    assert [x["c"] for x in r] == [13, 21, 34, 55, 89, 144, 233, 377, 610, 987]
    assert all(x["w"] == 0.0 for x in r)
    r = o.interp_rungs([10], 0.75, 0)  # d = 7.5: c = 8, position i - 7.5 = (i-8) + 0.5
    assert r[0]["c"] == 8 and r[0]["w"] == 0.5
    # fl64(alpha f) just below an integer: ceil picks that integer (kink reading)
    a5 = 0.5 + 5 / 15
    r = o.interp_rungs([144], a5, 8)
    assert r[0]["d"] < 120.0 and r[0]["c"] == 120


# ---------------------------------------------------------------- RoPE


def test_rope_equals_complex_rotation():
    """Rotate-half RoPE is multiplication of (x_j + i x_{j+D/2}) by e^{i t w_j}."""
    T, D, th = 37, 16, 1e4
    x = si.normal(3, T * D).reshape(T, D)
    cs, sn = o.rope_cos_sin(T, D, th)
    got = o.rope_apply(x, cs, sn)
    z = x[:, : D // 2] + 1j * x[:, D // 2 :]
    w = np.array([th ** (-2.0 * j / D) for j in range(D // 2)])
    zr = z * np.exp(1j * np.outer(np.arange(T), w))
    assert np.allclose(got[:, : D // 2], zr.real, atol=1e-12)
    assert np.allclose(got[:, D // 2 :], zr.imag, atol=1e-12)
    assert np.allclose(o.rope_apply(got, cs, sn, inverse=True), x, atol=1e-12)


def test_rope_relative_position():
    """q'(t1).k'(t2) depends only on t1 - t2."""
    T, D = 50, 8
    cs, sn = o.rope_cos_sin(T, D, 1e4)
    q = si.normal(4, D)
    k = si.normal(5, D)
    Q = o.rope_apply(np.tile(q, (T, 1)), cs, sn)
    Kr = o.rope_apply(np.tile(k, (T, 1)), cs, sn)
    assert abs(Q[20] @ Kr[13] - Q[40] @ Kr[33]) < 1e-12
    assert abs(Q[7] @ Kr[7] - q @ k) < 1e-12


# ---------------------------------------------------------------- forward pins


def _inputs(B, T, Hq, Hkv, D, seed=0):
    d = si.make_qkvdo(B, T, Hq, Hkv, D, "f32", seed)
    return {n: t.double().numpy() for n, t in d.items()}


def _dense_masked(q, k, v, allowed, theta):
    """Formulation (C): dense softmax with a boolean mask allowed[i, j]."""
    B, Hq, T, D = q.shape
    G = Hq // k.shape[1]
    if theta:
        cs, sn = o.rope_cos_sin(T, D, theta)
        q, k = o.rope_apply(q, cs, sn), o.rope_apply(k, cs, sn)
    O = np.zeros_like(q)
    for b in range(B):
        for h in range(Hq):
            S = q[b, h] @ k[b, h // G].T / math.sqrt(D)
            S = np.where(allowed, S, -np.inf)
            P = np.exp(S - S.max(1, keepdims=True))
            P /= P.sum(1, keepdims=True)
            O[b, h] = P @ v[b, h // G]
    return O


def _allowed_from_distances(T, dist):
    A = np.zeros((T, T), dtype=bool)
    for i in range(T):
        for s in dist:
            if 0 <= i - s:
                A[i, i - s] = True
    return A


@pytest.mark.parametrize("alpha,W", [(1.0, 3), (1.0, 0), (2.0 / 3.0, 2)])
def test_forward_integer_alpha_equals_boolean_mask(alpha, W):
    """At integer rung distances the lerp is an exact gather, so the result is
    the hard boolean-mask attention over window U rungs."""
    x = _inputs(2, 40, 4, 2, 8)
    base = [3, 6, 9, 15, 24]  # alpha*f integer for both alphas
    O, _ = o.forward(x["q"], x["k"], x["v"], o.interp_slots(base, alpha, W), 1e4)
    dist = set(range(W + 1)) | {round(alpha * f) for f in base}
    O2 = _dense_masked(x["q"], x["k"], x["v"], _allowed_from_distances(40, dist), 1e4)
    assert np.abs(O - O2).max() < 1e-12


def test_forward_int_slots_equal_boolean_mask_christoffel():
    x = _inputs(1, 70, 2, 2, 8)
    dist = o.christoffel_offsets(3, 8) + o.christoffel_offsets(3, 8, False)  # dup on purpose
    O, _ = o.forward(x["q"], x["k"], x["v"], o.dist_slots(dist), 0.0)
    O2 = _dense_masked(x["q"], x["k"], x["v"], _allowed_from_distances(70, set(dist)), 0.0)
    assert np.abs(O - O2).max() < 1e-12


def test_forward_general_alpha_equals_logit_lerp():
    """Formulation (B): the logit of a rung is the lerp of two dense logits
    at floor(i - d) and floor(i - d) + 1, and its probability is split over the
    two value rows with the same weights (the gather is linear)."""
    B, T, Hq, Hkv, D, W, alpha = 1, 45, 4, 2, 8, 2, 0.77
    x = _inputs(B, T, Hq, Hkv, D, 7)
    base = [1, 2, 3, 5, 8, 13, 21, 34]
    O, LSE = o.forward(x["q"], x["k"], x["v"], o.interp_slots(base, alpha, W), 1e4)
    cs, sn = o.rope_cos_sin(T, D, 1e4)
    q, k, v = o.rope_apply(x["q"], cs, sn), o.rope_apply(x["k"], cs, sn), x["v"]
    for h in range(Hq):
        g = h // (Hq // Hkv)
        S = q[0, h] @ k[0, g].T / math.sqrt(D)
        for i in range(T):
            logits, rows = [], []  # rows: list of [(row, weight)]
            for s in range(min(W, i) + 1):
                logits.append(S[i, i - s])
                rows.append([(i - s, 1.0)])
            for f in base:
                dk = alpha * f
                if dk <= W or dk > i:
                    continue
                x_pos = i - dk
                p0 = math.floor(x_pos)
                fr = x_pos - p0
                logits.append((1 - fr) * S[i, p0] + fr * S[i, p0 + 1])
                rows.append([(p0, 1 - fr), (p0 + 1, fr)])
            lg = np.array(logits)
            P = np.exp(lg - lg.max())
            lse = lg.max() + math.log(P.sum())
            P /= P.sum()
            out = np.zeros(D)
            for pe, rw in zip(P, rows):
                for r, wt in rw:
                    out += pe * wt * v[0, g, r]
            assert np.abs(out - O[0, h, i]).max() < 1e-12
            assert abs(lse - LSE[0, h, i]) < 1e-12


def test_forward_dense_special_case_and_T1():
    """W >= T-1 with no rungs is textbook causal softmax attention."""
    B, T, H, D = 1, 12, 2, 4
    x = _inputs(B, T, H, H, D, 11)
    O, _ = o.forward(x["q"], x["k"], x["v"], o.interp_slots([], 1.0, T - 1), 0.0)
    for h in range(H):
        Q, K, V = x["q"][0, h], x["k"][0, h], x["v"][0, h]
        want = np.zeros((T, D))
        for i in range(T):
            sc = np.array([Q[i] @ K[j] / 2.0 for j in range(i + 1)])
            p = np.exp(sc - sc.max())
            p /= p.sum()
            want[i] = sum(p[j] * V[j] for j in range(i + 1))
        assert np.abs(O[0, h] - want).max() < 1e-12
    x1 = _inputs(1, 1, 2, 1, 4, 12)
    O1, L1 = o.forward(x1["q"], x1["k"], x1["v"], o.interp_slots(o.fib_offsets(), 1.0, 8), 1e4)
    assert np.abs(O1[0, :, 0] - x1["v"][0, 0, 0][None]).max() < 1e-15


def test_forward_gqa_equals_repeated_kv():
    x = _inputs(1, 33, 8, 2, 8, 13)
    sl = o.interp_slots(o.fib_offsets(8), 0.9, 2)
    O, L = o.forward(x["q"], x["k"], x["v"], sl, 1e4)
    kr = np.repeat(x["k"], 4, axis=1)
    vr = np.repeat(x["v"], 4, axis=1)
    O2, L2 = o.forward(x["q"], kr, vr, sl, 1e4)
    assert np.abs(O - O2).max() < 1e-14 and np.abs(L - L2).max() < 1e-14


# ---------------------------------------------------------------- backward pins


def _loss(x, slots, theta, do):
    O, _ = o.forward(x["q"], x["k"], x["v"], slots, theta)
    return float(np.sum(O * do))


@pytest.mark.parametrize("alpha,W,theta", [(0.77, 1, 1e4), (1.0, 2, 0.0), (1.31, 0, 1e4)])
def test_backward_central_fd(alpha, W, theta):
    """Every element of dQ, dK, dV against central differences of L = sum O dO."""
    x = _inputs(1, 12, 4, 2, 4, 21)
    slots = o.interp_slots([1, 2, 3, 5, 8], alpha, W)
    g = o.backward(x["q"], x["k"], x["v"], x["do"], slots, theta)
    h = 1e-6
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv")):
        arr = x[name]
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + h
            lp = _loss(x, slots, theta, x["do"])
            arr[idx] = old - h
            lm = _loss(x, slots, theta, x["do"])
            arr[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        err = np.abs(num - g[key]).max() / max(1.0, np.abs(num).max())
        assert err < 1e-7, (name, err)


def _loss_alpha(x, base, alpha, W, theta):
    return _loss(x, o.interp_slots(base, alpha, W), theta, x["do"])


def test_dtheta_central_fd_away_from_kinks():
    x = _inputs(2, 40, 4, 2, 8, 23)
    base, W, th = [1, 2, 3, 5, 8, 13, 21, 34], 1, 0.3
    alpha = o.alpha_of_theta(th)
    frac = [abs(alpha * f - round(alpha * f)) for f in base]
    assert min(frac) > 1e-3
    g = o.backward(x["q"], x["k"], x["v"], x["do"], o.interp_slots(base, alpha, W), 1e4, alpha=alpha)
    h = 1e-7
    lp = _loss_alpha(x, base, o.alpha_of_theta(th + h), W, 1e4)
    lm = _loss_alpha(x, base, o.alpha_of_theta(th - h), W, 1e4)
    num = (lp - lm) / (2 * h)
    assert abs(num - g["dtheta"]) < 1e-6 * max(1.0, abs(num))
    # dalpha by itself, and the chain factor s(1 - s)
    ha = 1e-7
    na = (_loss_alpha(x, base, alpha + ha, W, 1e4) - _loss_alpha(x, base, alpha - ha, W, 1e4)) / (2 * ha)
    assert abs(na - g["dalpha"]) < 1e-6 * max(1.0, abs(na))
    s = 1.0 / (1.0 + math.exp(-th))
    assert abs(g["dtheta"] - g["dalpha"] * s * (1 - s)) < 1e-9 * max(1.0, abs(g["dtheta"]))


def test_dalpha_at_integer_alpha_is_left_derivative():
    """At alpha = 1 every rung sits on an integer (w = 0); the gradient that the
    interpolation keeps is the one-sided derivative from below in alpha."""
    x = _inputs(1, 40, 4, 2, 8, 29)
    base, W = [1, 2, 3, 5, 8, 13, 21], 1
    g = o.backward(x["q"], x["k"], x["v"], x["do"], o.interp_slots(base, 1.0, W), 1e4, alpha=1.0)
    assert abs(g["dalpha"]) > 1e-3  # nonzero even at integer positions
    h = 1e-7
    l0 = _loss_alpha(x, base, 1.0, W, 1e4)
    lm = _loss_alpha(x, base, 1.0 - h, W, 1e4)
    back = (l0 - lm) / h
    assert abs(back - g["dalpha"]) < 1e-5 * max(1.0, abs(back))


def test_backward_gqa_equals_repeated_kv_summed():
    x = _inputs(1, 20, 4, 2, 4, 31)
    sl = o.interp_slots([1, 2, 3, 5, 8, 13], 0.9, 1)
    g = o.backward(x["q"], x["k"], x["v"], x["do"], sl, 1e4)
    kr, vr = np.repeat(x["k"], 2, axis=1), np.repeat(x["v"], 2, axis=1)
    g2 = o.backward(x["q"], kr, vr, x["do"], sl, 1e4)
    assert np.abs(g["dq"] - g2["dq"]).max() < 1e-13
    assert np.abs(g["dk"] - g2["dk"].reshape(1, 2, 2, 20, 4).sum(2)).max() < 1e-13
    assert np.abs(g["dv"] - g2["dv"].reshape(1, 2, 2, 20, 4).sum(2)).max() < 1e-13


def test_dalpha_error_scales_bound_the_sum():
    """dalpha_abs / dalpha_rss (tolerance scales of the bf16 dL/dalpha check):
    |sum| <= sum of |terms| and rss <= sum of |terms| <= sqrt(#terms) rss."""
    x = si.make_qkvdo(1, 40, 4, 1, 64, "f32", seed=7)
    base = o.fib_offsets(8)
    g = o.backward(x["q"], x["k"], x["v"], x["do"], o.interp_slots(base, 0.9, 2), 1e4, alpha=0.9)
    n_terms = sum(2 * 40 * 64 for s in o.interp_slots(base, 0.9, 2) if s["kind"] == "rung")
    assert abs(g["dalpha"]) <= g["dalpha_abs"]
    assert 0.0 < g["dalpha_rss"] <= g["dalpha_abs"] <= math.sqrt(n_terms) * g["dalpha_rss"] * (1 + 1e-12)


def test_decode_is_the_forward_row_of_the_prefix():
    """oracle.decode at position t equals row t of the oracle forward over the
    prefix 0..t with the decode query placed at t (integer key set)."""
    B, T, Hq, Hkv = 2, 40, 4, 2
    x = si.make_qkvdo(B, T, Hq, Hkv, 8, "f32", seed=11, with_do=False)
    dist = o.int_distances(o.fib_offsets(8), 1.0, 3)
    pos = [39, 17]
    qd = x["q"][:, :, 0].numpy().astype(np.float64)
    O, L = o.decode(qd, x["k"], x["v"], pos, dist, 1e4)
    for b, t in enumerate(pos):
        qf = np.zeros((1, Hq, t + 1, 8))
        qf[0, :, t] = qd[b]
        Of, Lf = o.forward(qf, x["k"][b:b + 1, :, : t + 1], x["v"][b:b + 1, :, : t + 1],
                           o.dist_slots(dist), 1e4)
        np.testing.assert_allclose(O[b], Of[0, :, t], rtol=0, atol=1e-12)
        np.testing.assert_allclose(L[b], Lf[0, :, t], rtol=0, atol=1e-12)


def test_decode_dense_window_is_textbook_softmax():
    """With every distance 0..t present and no RoPE, decode is plain causal
    softmax attention of the last query over all cached rows (brute force)."""
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 2, 4))
    k = rng.standard_normal((1, 1, 6, 4))
    v = rng.standard_normal((1, 1, 6, 4))
    O, L = o.decode(q, k, v, [5], list(range(6)), 0.0)
    for h in range(2):
        s = [float(np.dot(q[0, h], k[0, 0, j])) / 2.0 for j in range(6)]
        w = [math.exp(x) for x in s]
        want = sum(w[j] * v[0, 0, j] for j in range(6)) / sum(w)
        np.testing.assert_allclose(O[0, h], want, rtol=0, atol=1e-12)
        assert abs(L[0, h] - math.log(sum(w))) < 1e-12


# ---- offset-schedule analysis and the shared power-law list ----------------


def test_reach_dense_window_closed_form():
    """L layers of the window {0..W}: d is reached after ceil(d / W) layers."""
    T, W, L = 200, 5, 7
    hops, covered = o.reach([list(range(W + 1))] * L, T)
    for d in range(T):
        want = -(-d // W) if -(-d // W) <= L else -1
        assert hops[d] == want, d
    assert covered == [min(T, l * W + 1) for l in range(1, L + 1)]


def test_reach_powers_of_two_is_popcount():
    """Layers {0, 1, 2, 4, ..., 2^k}: the fewest powers of two summing to d is
    popcount(d), so hops[d] = popcount(d) (d < 2^(k+1), within the stack)."""
    k, L = 6, 7
    T = 1 << (k + 1)
    S = [0] + [1 << j for j in range(k + 1)]
    hops, _ = o.reach([S] * L, T)
    for d in range(T):
        assert hops[d] == bin(d).count("1"), d


def test_reach_christoffel_residues():
    """Christoffel m/k = 128/1024 offsets {7, 15, ..., 1023} with 0: one layer
    reaches residues 0 and 7 mod 8 only; l layers reach residues
    {0, -1, ..., -l} mod 8, so 7 layers reach every class."""
    S = o.christoffel_offsets(128, 1024, include_zero=True)
    T = 2048
    for l in range(1, 9):
        hops, _ = o.reach([S] * l, T)
        cls = o.residue_classes(hops, 8)
        reached = {r for r in range(8) if cls[r] > 0}
        assert reached == {(-j) % 8 for j in range(l + 1)}, l


def test_offset_histogram_log2_bins():
    fib = [0, 1, 2, 3, 5, 8, 13, 21, 34, 55, 89, 89, 5000]
    assert o.offset_histogram(fib, 1024, 12) == [1, 1, 2, 1, 2, 1, 2, 1, 0, 0, 0, 0]
    assert o.offset_histogram([0, 600, 1023], 1024, 4) == [1, 0, 0, 2]


def test_powerlaw_extremes_and_invariants():
    n = 1024
    assert o.powerlaw_offsets([0.0], 0.8, n) == [1]
    assert o.powerlaw_offsets([1.0 - 2.0 ** -53], 0.8, n) == [n // 2]
    u = si.uniform(si.mix_seed(3, 1), 256)
    d = o.powerlaw_offsets(u, 0.85, n)
    assert d == sorted(set(d)) and 1 <= d[0] and d[-1] <= n // 2 and len(d) <= 256


def test_powerlaw_frequencies_follow_the_law():
    """Empirical frequencies of single draws match q(d) = d^-(1+s)/Z for the
    first distances (within 5 standard deviations of a binomial count)."""
    n, s, N = 1024, 0.8, 40000
    u = si.uniform(si.mix_seed(4, 2), N)
    Z = math.fsum(v ** -(1.0 + s) for v in range(1, n // 2 + 1))
    counts = {}
    for x in u:
        dd = o.powerlaw_offsets([x], s, n)[0]
        counts[dd] = counts.get(dd, 0) + 1
    for dd in (1, 2, 3, 10):
        p = dd ** -(1.0 + s) / Z
        assert abs(counts.get(dd, 0) - N * p) <= 5 * math.sqrt(N * p * (1 - p)), dd


# ---- signed offsets (bidirectional) ------------------------------------------


def test_signed_all_distances_is_full_softmax():
    """Distances -(T-1)..T-1, no RoPE: every query attends every key, the
    textbook full (non-causal) softmax attention, brute force."""
    x = _inputs(1, 7, 2, 1, 4, 31)
    O, L = o.forward(x["q"], x["k"], x["v"], o.dist_slots(range(-6, 7)), 0.0)
    for h in range(2):
        for t in range(7):
            s = [float(np.dot(x["q"][0, h, t], x["k"][0, 0, j])) / 2.0 for j in range(7)]
            m = max(s)
            w = [math.exp(v - m) for v in s]
            want = sum(w[j] * x["v"][0, 0, j] for j in range(7)) / sum(w)
            np.testing.assert_allclose(O[0, h, t], want, rtol=0, atol=1e-12)
            assert abs(L[0, h, t] - (m + math.log(sum(w)))) < 1e-12


def test_signed_time_reversal():
    """Without RoPE, reversing time maps distance s to -s: the forward of the
    reversed sequences with the negated set is the reversed forward."""
    x = _inputs(1, 20, 4, 2, 4, 33)
    S = [-7, -3, 0, 1, 2, 5, 11]
    O, L = o.forward(x["q"], x["k"], x["v"], o.dist_slots(S), 0.0)
    rev = {n: x[n][:, :, ::-1].copy() for n in ("q", "k", "v")}
    Or, Lr = o.forward(rev["q"], rev["k"], rev["v"], o.dist_slots([-s for s in S]), 0.0)
    np.testing.assert_allclose(Or[:, :, ::-1], O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(Lr[:, :, ::-1], L, rtol=0, atol=1e-12)


def test_signed_backward_central_fd():
    """dQ, dK, dV with future keys against central differences of L = sum O dO."""
    x = _inputs(1, 10, 4, 2, 4, 35)
    slots = o.dist_slots([-4, -1, 0, 2, 3])
    g = o.backward(x["q"], x["k"], x["v"], x["do"], slots, 1e4)
    h = 1e-6
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv")):
        arr = x[name]
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + h
            lp = _loss(x, slots, 1e4, x["do"])
            arr[idx] = old - h
            lm = _loss(x, slots, 1e4, x["do"])
            arr[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        err = np.abs(num - g[key]).max() / max(1.0, np.abs(num).max())
        assert err < 1e-7, (name, err)


def test_signed_christoffel_offsets():
    S = o.signed_christoffel_offsets(128, 1024)
    assert len(S) == 257 and S[127] == -7 and S[128] == 0 and S[129] == 7
    assert S == sorted(set(S)) and all(-x in S for x in S)
