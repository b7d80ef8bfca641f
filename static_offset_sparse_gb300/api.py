"""Python names for the libsfa C ABI (same names without the ``sfa_`` prefix).

Tensors are torch CUDA tensors, contiguous [B, H, T, 64], bf16 or fp32.  The
functions allocate outputs (and the backward workspace) with torch when they
are not given, take the current torch stream, and call the library.
"""
from __future__ import annotations

import ctypes as C

from ._lib import (SFA_BF16, SFA_F32, Desc, MAX_RUNGS, _lib, check, i32_array)

# ------------------------------------------------------------ host builders


def offsets_fib(K: int = 15) -> list[int]:
    out = (C.c_int32 * max(1, K))()
    check(_lib().sfa_offsets_fib(K, out), "sfa_offsets_fib")
    return list(out[:K])


def offsets_pow2(K: int = 11) -> list[int]:
    out = (C.c_int32 * max(1, K))()
    check(_lib().sfa_offsets_pow2(K, out), "sfa_offsets_pow2")
    return list(out[:K])


def offsets_christoffel(m: int, k: int, include_zero: bool = True) -> list[int]:
    n = C.c_int32(0)
    rc = _lib().sfa_offsets_christoffel(m, k, int(include_zero), None, 0, C.byref(n))
    if rc not in (0, 3):
        check(rc, "sfa_offsets_christoffel")
    out = (C.c_int32 * max(1, n.value))()
    check(_lib().sfa_offsets_christoffel(m, k, int(include_zero), out, n.value, C.byref(n)),
          "sfa_offsets_christoffel")
    return list(out[: n.value])


def alpha_schedule(L: int, kind: int, S: int = 7) -> list[float]:
    out = (C.c_double * max(1, L))()
    check(_lib().sfa_alpha_schedule(L, kind, S, out), "sfa_alpha_schedule")
    return list(out[:L])


def rung_table(base, alpha: float, W: int):
    """(c, w, f) lists of the interpolated path's rungs."""
    arr, n = i32_array(base)
    c = (C.c_int32 * MAX_RUNGS)()
    w = (C.c_float * MAX_RUNGS)()
    f = (C.c_float * MAX_RUNGS)()
    nout = C.c_int32(0)
    check(_lib().sfa_rung_table(arr, n, float(alpha), W, c, w, f, MAX_RUNGS, C.byref(nout)),
          "sfa_rung_table")
    k = nout.value
    return list(c[:k]), list(w[:k]), list(f[:k])


def int_distances(dist) -> list[int]:
    arr, n = i32_array(dist)
    out = (C.c_int32 * max(1, n))()
    nout = C.c_int32(0)
    check(_lib().sfa_int_distances(arr, n, out, max(1, n), C.byref(nout)), "sfa_int_distances")
    return list(out[: nout.value])


def band_plan(dist, T: int, G: int):
    """How the integer path lays a bf16 distance set out for the band
    kernels (sfa_band_plan): (delta, [(start, length), ...]); delta = 0 when
    the set runs the rung or SIMT kernels instead."""
    arr, n = i32_array(dist)
    cap = 256
    starts = (C.c_int32 * cap)()
    lens = (C.c_int32 * cap)()
    delta = C.c_int32(0)
    nruns = C.c_int32(0)
    check(_lib().sfa_band_plan(arr, n, T, G, C.byref(delta), starts, lens, cap, C.byref(nruns)),
          "sfa_band_plan")
    return delta.value, [(starts[m], lens[m]) for m in range(nruns.value)]


def reach(dist_sets, T: int):
    """Reachability through a stack of layers (sfa_reach): returns hops (list
    of T ints, -1 = never) and covered (one count per layer)."""
    flat = [int(x) for S in dist_sets for x in S]
    starts = [0]
    for S in dist_sets:
        starts.append(starts[-1] + len(S))
    darr, _ = i32_array(flat)
    sarr, _ = i32_array(starts)
    L = len(dist_sets)
    hops = (C.c_int32 * T)()
    cov = (C.c_int64 * max(1, L))()
    check(_lib().sfa_reach(darr, sarr, L, T, hops, cov), "sfa_reach")
    return list(hops), list(cov[:L])


def residue_classes(hops, M: int) -> list[int]:
    harr, T = i32_array(hops)
    out = (C.c_int64 * M)()
    check(_lib().sfa_residue_classes(harr, T, M, out), "sfa_residue_classes")
    return list(out)


def offset_histogram(dist, T: int, nb: int) -> list[int]:
    darr, n = i32_array(dist)
    out = (C.c_int64 * nb)()
    check(_lib().sfa_offset_histogram(darr, n, T, nb, out), "sfa_offset_histogram")
    return list(out)


def offsets_powerlaw(u, sigma: float, n: int) -> list[int]:
    """Shared power-law distances for the uniforms u (sfa_offsets_powerlaw)."""
    m = len(u)
    uarr = (C.c_double * max(1, m))(*[float(x) for x in u])
    out = (C.c_int32 * max(1, m))()
    nout = C.c_int32(0)
    check(_lib().sfa_offsets_powerlaw(uarr, m, float(sigma), int(n), out, max(1, m),
                                      C.byref(nout)), "sfa_offsets_powerlaw")
    return list(out[: nout.value])


def status_string(code: int) -> str:
    return _lib().sfa_status_string(code).decode()


# ------------------------------------------------------------ device calls

_ROPE_CACHE: dict = {}


def _torch():
    import torch

    return torch


def _stream():
    return C.c_void_p(_torch().cuda.current_stream().cuda_stream)


def rope_table(T: int, theta: float = 1e4, device=None):
    """fp32 [T, 32, 2] (cos, sin) table written by sfa_rope_table (cached)."""
    torch = _torch()
    dev = torch.device(device if device is not None else "cuda")
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    key = (int(T), float(theta), dev.index)
    tab = _ROPE_CACHE.get(key)
    if tab is None:
        tab = torch.empty((T, 32, 2), dtype=torch.float32, device=dev)
        with torch.cuda.device(dev):
            check(_lib().sfa_rope_table(T, float(theta), C.c_void_p(tab.data_ptr()), _stream()),
                  "sfa_rope_table")
        _ROPE_CACHE[key] = tab
    return tab


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return SFA_BF16
    if t.dtype == torch.float32:
        return SFA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _check_tensor(t, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (libsfa has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def make_desc(q, k, *, W=0, alpha=1.0, base=(), dist=(), rope_theta=1e4, k_rot=None):
    """Build the sfa_desc for k [B,Hkv,T,64] and q [B,Hq,...] (Hq and the
    dtype are taken from q).  Keeps the host arrays alive on the returned
    object."""
    B, Hkv, T, D = k.shape
    Hq = q.shape[1]
    d = Desc()
    d.B, d.T, d.Hq, d.Hkv, d.D = B, T, Hq, Hkv, D
    d.dtype = _dtype_code(q)
    d.W = int(W)
    d.alpha = float(alpha)
    barr, nb = i32_array(base)
    darr, nd = i32_array(dist)
    d.base, d.n_base = C.cast(barr, C.POINTER(C.c_int32)), nb
    d.dist, d.n_dist = C.cast(darr, C.POINTER(C.c_int32)), nd
    if rope_theta and rope_theta > 0:
        tab = rope_table(T, rope_theta, q.device)
        d.rope = C.c_void_p(tab.data_ptr())
        d._keep = (barr, darr, tab)
    else:
        d.rope = None
        d._keep = (barr, darr)
    d.k_rot = C.c_void_p(k_rot.data_ptr()) if k_rot is not None else None
    d._keep = d._keep + ((k_rot,) if k_rot is not None else ())
    return d


def _ptr(t):
    return C.c_void_p(t.data_ptr()) if t is not None else None


def workspace_size(desc, interp: bool = True, backward: bool = True) -> int:
    n = C.c_size_t(0)
    check(_lib().sfa_workspace_size(C.byref(desc), int(interp), int(backward), C.byref(n)),
          "sfa_workspace_size")
    return n.value


def _workspace(desc, interp, backward, device, ws=None):
    n = workspace_size(desc, interp, backward)
    if ws is None or ws.numel() < n:
        ws = _torch().empty((max(n, 1),), dtype=_torch().uint8, device=device)
    return ws, n


def _fwd(fn, name, interp, q, k, v, desc, o=None, lse=None, ws=None):
    torch = _torch()
    for t, nm in ((q, "q"), (k, "k"), (v, "v")):
        _check_tensor(t, nm)
    B, Hq, T, _ = q.shape
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device)
    ws, n = _workspace(desc, interp, False, q.device, ws)
    check(fn(C.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(ws), n, _stream()),
          name)
    return o, lse


def forward(q, k, v, *, W: int, alpha: float, base, rope_theta: float = 1e4, o=None, lse=None,
            ws=None, k_rot=None):
    """Interpolated path: window 0..W plus rungs alpha*f for f in base.  k_rot:
    optional rotated keys from rope_keys (skips the call's own rotation)."""
    desc = make_desc(q, k, W=W, alpha=alpha, base=base, rope_theta=rope_theta, k_rot=k_rot)
    return _fwd(_lib().sfa_forward, "sfa_forward", True, q, k, v, desc, o, lse, ws)


def forward_int(q, k, v, *, dist, rope_theta: float = 1e4, o=None, lse=None, ws=None, k_rot=None):
    """Integer path: keys i - s for s in dist (0 required)."""
    desc = make_desc(q, k, dist=dist, rope_theta=rope_theta, k_rot=k_rot)
    return _fwd(_lib().sfa_forward_int, "sfa_forward_int", False, q, k, v, desc, o, lse, ws)


def _bwd(interp, q, k, v, o, lse, do, desc, dq=None, dk=None, dv=None, ws=None, dadt=None):
    torch = _torch()
    for t, nm in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (lse, "lse"), (do, "do")):
        _check_tensor(t, nm)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws, nws = _workspace(desc, interp, True, q.device, ws)
    L = _lib()
    if interp:
        if dadt is None:
            dadt = torch.empty((2,), dtype=torch.float64, device=q.device)
        check(L.sfa_backward(C.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                             _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dadt), _ptr(ws),
                             nws, _stream()), "sfa_backward")
        return dq, dk, dv, dadt
    check(L.sfa_backward_int(C.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                             _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), nws, _stream()),
          "sfa_backward_int")
    return dq, dk, dv


def backward(q, k, v, o, lse, do, *, W: int, alpha: float, base, rope_theta: float = 1e4,
             k_rot=None, **out):
    """Returns dq, dk, dv and a device float64 [2] tensor (dL/dalpha, dL/dtheta)."""
    desc = make_desc(q, k, W=W, alpha=alpha, base=base, rope_theta=rope_theta, k_rot=k_rot)
    return _bwd(True, q, k, v, o, lse, do, desc, **out)


def backward_int(q, k, v, o, lse, do, *, dist, rope_theta: float = 1e4, k_rot=None, **out):
    desc = make_desc(q, k, dist=dist, rope_theta=rope_theta, k_rot=k_rot)
    return _bwd(False, q, k, v, o, lse, do, desc, **out)


def rope_keys(k, rope_theta: float = 1e4, out=None):
    """Rotated keys for the k_rot argument (sfa_rope_keys; bf16)."""
    _check_tensor(k, "k")
    desc = make_desc(k, k, rope_theta=rope_theta)
    out = _torch().empty_like(k) if out is None else out
    check(_lib().sfa_rope_keys(C.byref(desc), _ptr(k), _ptr(out), _stream()), "sfa_rope_keys")
    return out


def decode_int(q, k_cache, v_cache, pos, *, dist, rope_theta: float = 1e4, o=None, lse=None):
    """One decode step on the integer path: q [B, Hq, 64] at positions pos
    (int32 [B], on the device) against caches [B, Hkv, T, 64] (raw keys).
    Returns o [B, Hq, 64] and lse fp32 [B, Hq]."""
    torch = _torch()
    for t, nm in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (pos, "pos")):
        _check_tensor(t, nm)
    if q.dim() != 3 or k_cache.dim() != 4 or pos.dtype != torch.int32:
        raise ValueError("decode_int: q [B, Hq, 64], caches [B, Hkv, T, 64], pos int32 [B]")
    B, Hkv, T, D = k_cache.shape
    desc = make_desc(q, k_cache, dist=dist, rope_theta=rope_theta)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, q.shape[1]), dtype=torch.float32, device=q.device) if lse is None else lse
    check(_lib().sfa_decode_int(C.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(pos),
                                _ptr(o), _ptr(lse), _stream()), "sfa_decode_int")
    return o, lse


def get_device_status() -> int:
    out = C.c_int32(0)
    check(_lib().sfa_get_device_status(_stream(), C.byref(out)), "sfa_get_device_status")
    return out.value


KERNEL_KINDS = ("fwd", "bwd_q", "bwd_kv", "dalpha_reduce", "rope_table", "prep", "decode")


def timing_enable(on: bool = True) -> None:
    """Bracket every library kernel launch with CUDA events on its stream."""
    check(_lib().sfa_timing_enable(int(on)), "sfa_timing_enable")


def timing_read() -> dict:
    """{kernel kind: (total ms, launches)} since the last read."""
    n = len(KERNEL_KINDS)
    ms = (C.c_double * n)()
    cnt = (C.c_int64 * n)()
    check(_lib().sfa_timing_read(ms, cnt, n), "sfa_timing_read")
    return {k: (ms[i], cnt[i]) for i, k in enumerate(KERNEL_KINDS)}
