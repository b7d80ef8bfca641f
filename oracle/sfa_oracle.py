"""Plain fp64 definition of causal shared-offset sparse attention (the oracle).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the library.  No code is
shared with the CUDA path.

Sources (page title, then the part of the page):
  [FIB]  "Depth-Staggered Fibonacci Spacing for Sparse Attention", method
         section: key set = window {0..W} union scaled Fibonacci rungs
         d_k = alpha * f_k; rung rows gathered by linear interpolation between
         the floor and floor-plus-one positions; RoPE at true positions before
         the gather; alpha = 0.5 + sigmoid(theta); the four layer schedules; the
         power-of-2 control; the fused boolean-mask path for integer offsets.
  [FIB-setup] same page, setup: GQA 8 query / 2 KV heads, head dim 64,
         RoPE theta 1e4, T = 1024.
  [CHR]  "Christoffel-Balanced Sparse Attention": carry word
         c[j] = floor((j+1)m/k) - floor(jm/k), offsets O = {j : c[j] = 1},
         causal keys, logits scaled by 1/sqrt(d).

Every function computes the plain definition with numpy in fp64.  Readings
where the pages are silent are stated next to the code that takes them.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, printed values, brute force, finite differences); none is
"parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np

# --------------------------------------------------------------------------
# offset lists
# --------------------------------------------------------------------------


def fib_offsets(K: int = 15) -> list[int]:
    """First K terms of the base sequence 1, 2, 3, 5, 8, ... [FIB, method].

    Each term is the sum of the previous two, starting from 1, 2.
    """
    if K < 1:
        raise ValueError("K >= 1")
    out = [1, 2]
    while len(out) < K:
        out.append(out[-1] + out[-2])
    return out[:K]


def pow2_offsets(K: int = 11) -> list[int]:
    """Power-of-2 control base 1, 2, 4, ..., 2^(K-1) [FIB, method, control].

    The page names a reach-matched log-sparse base; 11 terms reach 1024.
    """
    if K < 1:
        raise ValueError("K >= 1")
    return [1 << j for j in range(K)]


def christoffel_word(m: int, k: int) -> list[int]:
    """Carry word c[j] = floor((j+1)m/k) - floor(jm/k), j = 0..k-1 [CHR].

    Python integers are exact, so this is the integer arithmetic the page asks
    for.
    """
    if not (0 < m <= k):
        raise ValueError("0 < m <= k")
    return [((j + 1) * m) // k - (j * m) // k for j in range(k)]


def christoffel_offsets(m: int, k: int, include_zero: bool = True) -> list[int]:
    """Allowed offsets O = {j : c[j] = 1}, plus 0 when asked [CHR].

    Reading: query i attends keys i - o for o in O (kept when >= 0); the
    self-distance 0 is added so no row is empty.  Sorted ascending.
    """
    c = christoffel_word(m, k)
    o = [j for j, cj in enumerate(c) if cj == 1]
    if include_zero and 0 not in o:
        o = [0] + o
    return sorted(o)


# --------------------------------------------------------------------------
# alpha schedules [FIB, method]
# --------------------------------------------------------------------------

SCHED_FIXED, SCHED_LINEAR, SCHED_COPRIME = 0, 1, 2


def alpha_of_theta(theta: float) -> float:
    """alpha = 0.5 + sigmoid(theta), in [0.5, 1.5]."""
    return 0.5 + 1.0 / (1.0 + math.exp(-theta))


def theta_of_alpha(alpha: float) -> float:
    """Inverse of alpha_of_theta; +-inf at the ends of [0.5, 1.5]."""
    s = alpha - 0.5
    if s <= 0.0:
        return -math.inf
    if s >= 1.0:
        return math.inf
    return math.log(s / (1.0 - s))


def alpha_schedule(L: int, kind: int, S: int = 7) -> list[float]:
    """Per-layer alpha for the fixed, linear and coprime (HDC) schedules.

    fixed:   alpha_l = 1.
    linear:  alpha_l = 0.5 + l/(L-1).
    coprime: the linear multiset reassigned by l -> S*l mod L, i.e. layer l
             takes the linear value of index (S*l mod L).  Requires gcd(S,L)=1.
    """
    if L < 1:
        raise ValueError("L >= 1")
    if kind == SCHED_FIXED:
        return [1.0] * L
    lin = [0.5 + l / (L - 1) if L > 1 else 1.0 for l in range(L)]
    if kind == SCHED_LINEAR:
        return lin
    if kind == SCHED_COPRIME:
        if math.gcd(S, L) != 1:
            raise ValueError("gcd(S, L) must be 1")
        return [lin[(S * l) % L] for l in range(L)]
    raise ValueError("unknown schedule kind")


# --------------------------------------------------------------------------
# rung tables and key slots [FIB, method]
# --------------------------------------------------------------------------


def interp_rungs(base, alpha: float, W: int) -> list[dict]:
    """Interpolated rungs for one layer.

    d_k = fl64(alpha * f_k).  Reading (the key set is a *union* with the
    window): a rung with d_k <= W lies inside the window and is dropped.  For a
    kept rung, c_k = ceil(d_k) and w_k = c_k - d_k in [0, 1): the row at real
    position i - d_k is (1 - w_k) * row[i - c_k] + w_k * row[i - c_k + 1], the
    floor / floor-plus-one interpolation of the page.
    """
    out = []
    for f in base:
        d = float(alpha) * float(f)
        if d <= W:
            continue
        c = math.ceil(d)
        out.append({"f": float(f), "d": d, "c": int(c), "w": c - d})
    return out


def int_distances(base, alpha: float, W: int) -> list[int]:
    """Integer-offset key distances {0..W} union {round(alpha f_k)}.

    Reading: rounding is round-half-to-even (Python ``round``) of fl64(alpha
    f_k); duplicates collapse (a set union).
    """
    s = set(range(W + 1))
    for f in base:
        s.add(int(round(float(alpha) * float(f))))
    return sorted(s)


def window_slots(W: int) -> list[dict]:
    return [{"kind": "win", "s": s} for s in range(W + 1)]


def rung_slots(rungs) -> list[dict]:
    return [{"kind": "rung", "c": r["c"], "w": r["w"], "f": r["f"]} for r in rungs]


def dist_slots(dist) -> list[dict]:
    """Integer path: one exact-gather slot per distance (negative = future key)."""
    return [{"kind": "win", "s": int(s)} for s in sorted(set(int(x) for x in dist))]


def signed_christoffel_offsets(m: int, k: int) -> list[int]:
    """Signed offsets for bidirectional attention ("Christoffel-Balanced
    Sparse Attention": use signed offsets): the carry-word offsets O and
    their negatives, with 0 (self) once."""
    O = christoffel_offsets(m, k, include_zero=True)
    return sorted(set(O) | {-x for x in O})


def interp_slots(base, alpha: float, W: int) -> list[dict]:
    return window_slots(W) + rung_slots(interp_rungs(base, alpha, W))


# --------------------------------------------------------------------------
# RoPE [FIB, method (rotation at each row's own position, ahead of the gather); FIB-setup]
# --------------------------------------------------------------------------


def rope_cos_sin(T: int, D: int, theta: float):
    """cos/sin of phi(t, j) = t * theta^(-2j/D), t < T, j < D/2, fp64.

    Reading: rotate-half pairing (j, j + D/2).
    """
    j = np.arange(D // 2, dtype=np.float64)
    inv = theta ** (-(2.0 * j) / D)
    ang = np.arange(T, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang), np.sin(ang)


def rope_apply(x, cos, sin, inverse: bool = False):
    """Rotate the last dim of x [..., T, D] by +phi (or -phi if inverse)."""
    h = x.shape[-1] // 2
    a, b = x[..., :h], x[..., h:]
    s = -sin if inverse else sin
    return np.concatenate([a * cos - b * s, a * s + b * cos], axis=-1)


# --------------------------------------------------------------------------
# attention forward / backward [FIB, method; CHR for the 1/sqrt(d) scale]
# --------------------------------------------------------------------------


def _as64(x):
    if hasattr(x, "detach"):  # torch tensor (any dtype) -> fp64 numpy
        import torch

        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def _slot_rows(kr, v, slots, T):
    """Key/value row seen by every query t through every slot, for one KV head.

    kr, v: [T, D] (kr already rotated).  Returns Ks, Vs [n, T, D] and the
    validity mask [n, T].  Window / integer slot s: row t - s, valid iff
    0 <= t - s < T (a negative s, from a signed offset list, reads the
    future row t + |s|: "Christoffel-Balanced Sparse Attention", signed
    offsets for bidirectional attention).  Rung (c, w): (1-w) row[t-c] +
    w row[t-c+1], valid iff t >= c (i.e. d_k <= t; the rung is absent for
    earlier queries).
    """
    n, D = len(slots), kr.shape[-1]
    Ks = np.zeros((n, T, D))
    Vs = np.zeros((n, T, D))
    ok = np.zeros((n, T), dtype=bool)
    for a, sl in enumerate(slots):
        if sl["kind"] == "win":
            s = sl["s"]
            if abs(s) >= T:
                continue
            if s >= 0:
                Ks[a, s:] = kr[: T - s]
                Vs[a, s:] = v[: T - s]
                ok[a, s:] = True
            else:  # query t reads row t + |s| while it exists
                Ks[a, : T + s] = kr[-s:]
                Vs[a, : T + s] = v[-s:]
                ok[a, : T + s] = True
        else:
            c, w = sl["c"], sl["w"]
            if c >= T:
                continue
            Ks[a, c:] = (1.0 - w) * kr[: T - c] + w * kr[1 : T - c + 1]
            Vs[a, c:] = (1.0 - w) * v[: T - c] + w * v[1 : T - c + 1]
            ok[a, c:] = True
    return Ks, Vs, ok


def forward(q, k, v, slots, rope_theta: float = 1e4, rows=None):
    """O [B,Hq,T,D] and LSE [B,Hq,T] (fp64) for the given key slots.

    q [B,Hq,T,D], k/v [B,Hkv,T,D].  Query head h reads KV head h // (Hq/Hkv)
    (reading: contiguous GQA groups).  RoPE (rope_theta > 0) rotates q and k at
    their own positions before the slot gather; v is not rotated.  Logits are
    q'.k / sqrt(D); softmax over the valid slots; O = sum P v.
    ``rows`` optionally restricts the work to a list of (b, kv_head) pairs
    (the other entries of the result are left as NaN).
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(D)
    if rope_theta and rope_theta > 0:
        cs, sn = rope_cos_sin(T, D, rope_theta)
        q, k = rope_apply(q, cs, sn), rope_apply(k, cs, sn)
    O = np.full((B, Hq, T, D), np.nan)
    LSE = np.full((B, Hq, T), np.nan)
    pairs = rows if rows is not None else [(b, g) for b in range(B) for g in range(Hkv)]
    for b, g in pairs:
        Ks, Vs, ok = _slot_rows(k[b, g], v[b, g], slots, T)
        for h in range(g * G, (g + 1) * G):
            s = np.einsum("td,ntd->nt", q[b, h], Ks) * scale
            s = np.where(ok, s, -np.inf)
            m = s.max(axis=0)
            e = np.exp(s - m)
            l = e.sum(axis=0)
            P = e / l
            O[b, h] = np.einsum("nt,ntd->td", P, Vs)
            LSE[b, h] = m + np.log(l)
    return O, LSE


def decode(q, k, v, pos, dist, rope_theta: float = 1e4):
    """One decode step on the integer path (fp64).

    q [B,Hq,D]: the query of sequence b at position pos[b]; k/v [B,Hkv,T,D]:
    the caches (raw keys).  Keys of sequence b: pos[b] - s for s in dist with
    s <= pos[b] ("Depth-Staggered ...", method section: integer offsets as an
    exact gather).  RoPE rotates the query at pos[b] and every key at its own
    position; logits q'.k' / sqrt(D), softmax, O = sum P v.  Returns O
    [B,Hq,D] and LSE [B,Hq]: the forward's row pos[b] of that prefix.
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, Hq, D = q.shape
    Hkv, T = k.shape[1], k.shape[2]
    G = Hq // Hkv
    S = sorted({int(x) for x in dist})
    rot = bool(rope_theta and rope_theta > 0)
    if rot:
        cs, sn = rope_cos_sin(T, D, rope_theta)
    O = np.zeros((B, Hq, D))
    LSE = np.zeros((B, Hq))
    for b in range(B):
        t = int(pos[b])
        keys = np.array([t - x for x in S if x <= t], dtype=np.int64)
        for h in range(Hq):
            g = h // G
            qh, Kr = q[b, h], k[b, g, keys]
            if rot:
                qh = rope_apply(qh[None], cs[t:t + 1], sn[t:t + 1])[0]
                Kr = rope_apply(Kr, cs[keys], sn[keys])
            sc = Kr @ qh / math.sqrt(D)
            m = sc.max()
            e = np.exp(sc - m)
            O[b, h] = (e / e.sum()) @ v[b, g, keys]
            LSE[b, h] = m + math.log(e.sum())
    return O, LSE


def backward(q, k, v, do, slots, rope_theta: float = 1e4, alpha: float | None = None, rows=None):
    """Gradients of L = sum(O * dO) (no batch averaging).

    ``rows`` optionally restricts the work to a list of (b, kv_head) pairs:
    only their dq / dk / dv entries are computed (others stay 0) and dd,
    dalpha, dtheta then sum over those pairs only.

    Returns a dict with dq, dk, dv (fp64, the inputs' shapes), dd (one entry
    per rung slot: dL/dd_k) and, when ``alpha`` is given, dalpha and dtheta.
    dd_abs / dalpha_abs are the same sums taken over the absolute values of
    their (position, dimension) terms, and dalpha_rss the root of the sum of
    their squares: the scales of the rounding error of a low-precision
    evaluation of dalpha, whose terms cancel.

    Per query t and slot n (P, O from the forward):
      delta = dO . O;  dP = dO . v_n;  dS = P (dP - delta)
      dq' = sum_n dS k_n / sqrt(D)
      a window slot scatters dS q'/sqrt(D) to key row t-s and P dO to value
      row t-s; a rung (c, w) scatters them with weights (1-w) to row t-c and w
      to row t-c+1 (the gather is linear in the two rows).
      dL/dd_k = sum dS q'.(k'[t-c] - k'[t-c+1]) / sqrt(D)
                + P dO.(v[t-c] - v[t-c+1])
      (c is held fixed and w = c - d, so d(row)/dd = row[t-c] - row[t-c+1]:
      the left derivative at an integer d).
      dQ = R(-phi) dq', dK = R(-phi) dk' (V is not rotated).
      dalpha = sum_k f_k dL/dd_k (d_k = alpha f_k);
      dtheta = dalpha * s (1 - s), s = sigmoid(theta) = alpha - 0.5.
    """
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(D)
    rot = bool(rope_theta and rope_theta > 0)
    if rot:
        cs, sn = rope_cos_sin(T, D, rope_theta)
        q, k = rope_apply(q, cs, sn), rope_apply(k, cs, sn)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    rung_ids = [a for a, sl in enumerate(slots) if sl["kind"] == "rung"]
    dd = np.zeros(len(rung_ids))
    dd_abs = np.zeros(len(rung_ids))
    dd_sq = np.zeros(len(rung_ids))
    pairs = rows if rows is not None else [(b, g) for b in range(B) for g in range(Hkv)]
    for b, g in pairs:
        Ks, Vs, ok = _slot_rows(k[b, g], v[b, g], slots, T)
        dKs = np.zeros_like(Ks)
        dVs = np.zeros_like(Vs)
        for h in range(g * G, (g + 1) * G):
            s = np.where(ok, np.einsum("td,ntd->nt", q[b, h], Ks) * scale, -np.inf)
            m = s.max(axis=0)
            e = np.exp(s - m)
            P = e / e.sum(axis=0)
            O = np.einsum("nt,ntd->td", P, Vs)
            delta = np.einsum("td,td->t", do[b, h], O)
            dP = np.einsum("td,ntd->nt", do[b, h], Vs)
            dS = np.where(ok, P * (dP - delta), 0.0)
            dq[b, h] = np.einsum("nt,ntd->td", dS, Ks) * scale
            dKs += dS[:, :, None] * q[b, h][None] * scale
            dVs += P[:, :, None] * do[b, h][None]
        for a, sl in enumerate(slots):
            if sl["kind"] == "win":
                s_ = sl["s"]
                if abs(s_) >= T:
                    continue
                if s_ >= 0:
                    dk[b, g, : T - s_] += dKs[a, s_:]
                    dv[b, g, : T - s_] += dVs[a, s_:]
                else:  # key row t + |s| collects from query t
                    dk[b, g, -s_:] += dKs[a, : T + s_]
                    dv[b, g, -s_:] += dVs[a, : T + s_]
            else:
                c, w = sl["c"], sl["w"]
                if c >= T:
                    continue
                dk[b, g, : T - c] += (1.0 - w) * dKs[a, c:]
                dk[b, g, 1 : T - c + 1] += w * dKs[a, c:]
                dv[b, g, : T - c] += (1.0 - w) * dVs[a, c:]
                dv[b, g, 1 : T - c + 1] += w * dVs[a, c:]
                r = rung_ids.index(a)
                dK_row = k[b, g, : T - c] - k[b, g, 1 : T - c + 1]
                dV_row = v[b, g, : T - c] - v[b, g, 1 : T - c + 1]
                tk, tv = dKs[a, c:] * dK_row, dVs[a, c:] * dV_row
                dd[r] += np.sum(tk) + np.sum(tv)
                dd_abs[r] += np.sum(np.abs(tk)) + np.sum(np.abs(tv))
                dd_sq[r] += np.sum(tk * tk) + np.sum(tv * tv)
    if rot:
        dq = rope_apply(dq, cs, sn, inverse=True)
        dk = rope_apply(dk, cs, sn, inverse=True)
    out = {"dq": dq, "dk": dk, "dv": dv, "dd": dd, "dd_abs": dd_abs}
    if alpha is not None:
        f = np.array([slots[a]["f"] for a in rung_ids])
        dalpha = float(np.sum(f * dd))
        out["dalpha"] = dalpha
        out["dalpha_abs"] = float(np.sum(np.abs(f) * dd_abs))
        out["dalpha_rss"] = float(math.sqrt(np.sum(f * f * dd_sq)))
        out["dtheta"] = dalpha * (alpha - 0.5) * (1.5 - alpha)
    return out


# --------------------------------------------------------------------------
# offset-schedule analysis and the shared power-law offset list
# --------------------------------------------------------------------------


def reach(dist_sets, T: int):
    """Distances reached through a stack of causal shared-offset layers.

    ("Christoffel-Balanced Sparse Attention": measure graph reachability
    across layers, since a single periodic mask may leave residue classes
    unreached; "Depth-Staggered ...": coverage through the stack.)  Layer l
    lets position i read position i - s for s in dist_sets[l] (s >= 0).  After
    layers 1..l, distance d is reached iff d = s_1 + ... + s_l with s_j in
    dist_sets[j - 1] and d < T; before any layer only d = 0 is.

    Returns (hops, covered): hops[d] = the smallest l >= 0 after which d is
    reached (-1 if never within the stack), covered[l - 1] = the number of
    distances < T reached after exactly layers 1..l.
    """
    R = {0}
    hops = [-1] * T
    hops[0] = 0
    covered = []
    for l, S in enumerate(dist_sets, start=1):
        R = {r + s for r in R for s in S if r + s < T}
        for d in R:
            if hops[d] < 0:
                hops[d] = l
        covered.append(len(R))
    return hops, covered


def residue_classes(hops, M: int):
    """Number of reached distances (hops >= 0) in each residue class mod M."""
    out = [0] * M
    for d, h in enumerate(hops):
        if h >= 0:
            out[d % M] += 1
    return out


def offset_histogram(dist, T: int, nb: int):
    """Histogram of a distance set (duplicates counted once, d < T only) in
    log2 bins: bin 0 = {0}; bin b = [2^(b-1), 2^b) for 1 <= b < nb - 1; the
    last bin takes every d >= 2^(nb-2)."""
    h = [0] * nb
    for d in sorted(set(int(x) for x in dist)):
        if d < 0 or d >= T:
            continue
        if d == 0:
            b = 0
        else:
            b = min(nb - 1, d.bit_length())
        h[b] += 1
    return h


def powerlaw_offsets(u, sigma: float, n: int):
    """Shared power-law offset list ("Critical power-law sparse attention",
    integration point: the fixed-degree approximation draws m distances from
    q(d) = d^-(1+sigma) / sum_{v=1}^{floor(n/2)} v^-(1+sigma), d = 1..floor(n/2),
    and deduplicates).  Here one draw serves every query (shared offsets,
    causal keys i - d); u holds the m uniforms in [0, 1).

    Inverse CDF in fp64: c_d = sum_{v<=d} v^-(1+sigma) summed in increasing v,
    Z = c_{floor(n/2)}; draw j takes the smallest d with c_d > u_j * Z.
    Returns the distinct distances, ascending.
    """
    Dmax = n // 2
    c = []
    acc = 0.0
    for v in range(1, Dmax + 1):
        acc += float(v) ** (-(1.0 + sigma))
        c.append(acc)
    Z = c[-1]
    out = set()
    for x in u:
        t = float(x) * Z
        lo, hi = 0, Dmax - 1  # smallest index with c[idx] > t
        while lo < hi:
            mid = (lo + hi) // 2
            if c[mid] > t:
                hi = mid
            else:
                lo = mid + 1
        out.add(lo + 1)
    return sorted(out)
