"""Seeded synthetic inputs shared by the oracle and the CUDA path.

This module draws random numbers and rounds them to the storage dtype; it holds
none of the attention arithmetic, so both the fp64 oracle (``oracle/``) and the
GPU tests / benchmark can use it without sharing any of the method's code.

Generator (fully specified, platform independent):
  * SplitMix64 (Steele, Lea, Flood 2014; constants as published by Vigna):
    the n-th output of stream ``s`` is ``mix(s + (n + 1) * 0x9E3779B97F4A7C15)``.
  * 53-bit uniforms ``u = (z >> 11) * 2**-53`` in [0, 1).
  * Box-Muller in fp64: ``r = sqrt(-2 ln(1 - u0))``, ``n0 = r cos(2 pi u1)``,
    ``n1 = r sin(2 pi u1)`` from consecutive uniform pairs.
  * Rounded to the storage dtype with round-to-nearest-even (through fp32 for
    bf16; the rounded values are what both sides consume).

The workloads on the pages draw Q, K, V and dO i.i.d. N(0, 1); tensors use the
[B, H, T, D] contiguous layout.
"""
from __future__ import annotations

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# tensor ids used when mixing a seed for one tensor of one layer
TENSOR_IDS = {"q": 1, "k": 2, "v": 3, "do": 4}


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(seed: int, n: int, start: int = 0) -> np.ndarray:
    """Outputs ``start .. start+n-1`` of the SplitMix64 stream seeded with ``seed``."""
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        state = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * _GAMMA
        return _mix(state)


def mix_seed(seed: int, *ids: int) -> int:
    """Derive an independent stream seed from a base seed and integer ids."""
    s = seed & 0xFFFFFFFFFFFFFFFF
    for i in ids:
        s = int(splitmix64(s ^ ((i * 0x2545F4914F6CDD1D) & 0xFFFFFFFFFFFFFFFF), 1)[0])
    return s


def uniform(seed: int, n: int) -> np.ndarray:
    z = splitmix64(seed, n)
    return (z >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def normal(seed: int, n: int) -> np.ndarray:
    """``n`` i.i.d. N(0, 1) draws in fp64 (Box-Muller on SplitMix64 uniforms)."""
    m = (n + 1) // 2
    u = uniform(seed, 2 * m)
    r = np.sqrt(-2.0 * np.log1p(-u[0::2]))
    t = 2.0 * np.pi * u[1::2]
    out = np.empty(2 * m, dtype=np.float64)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.sin(t)
    return out[:n]


def round_to(x: np.ndarray, dtype: str):
    """Round fp64 values to the storage dtype; returns a torch CPU tensor.

    ``dtype`` is ``"f32"`` or ``"bf16"``.  bf16 goes fp64 -> fp32 -> bf16, both
    steps round-to-nearest-even.
    """
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    if dtype == "f32":
        return t
    if dtype == "bf16":
        return t.to(torch.bfloat16)
    raise ValueError(f"unknown dtype {dtype!r}")


def make_tensor(shape, dtype: str, seed: int, *ids: int):
    """One N(0, 1) tensor of ``shape`` (row-major), seeded by ``(seed, *ids)``."""
    n = int(np.prod(shape))
    x = normal(mix_seed(seed, *ids), n).reshape(shape)
    return round_to(x, dtype)


def make_qkvdo(B: int, T: int, Hq: int, Hkv: int, D: int, dtype: str,
               seed: int, layer: int = 0, with_do: bool = True):
    """Q [B,Hq,T,D], K/V [B,Hkv,T,D] and (optionally) dO [B,Hq,T,D] on the host.

    Fill order is Q, K, V, dO; each tensor has its own stream derived from
    ``(seed, layer, tensor id)``.
    """
    out = {
        "q": make_tensor((B, Hq, T, D), dtype, seed, layer, TENSOR_IDS["q"]),
        "k": make_tensor((B, Hkv, T, D), dtype, seed, layer, TENSOR_IDS["k"]),
        "v": make_tensor((B, Hkv, T, D), dtype, seed, layer, TENSOR_IDS["v"]),
    }
    if with_do:
        out["do"] = make_tensor((B, Hq, T, D), dtype, seed, layer, TENSOR_IDS["do"])
    return out


# ---------------------------------------------------------------- on device
#
# The same stream computed with torch integer ops on a device (used by the
# benchmark, where host generation of gigabytes would dominate the run).  The
# integer stream is bit-identical to ``splitmix64``; the fp64 Box-Muller may
# differ from numpy's by an ulp of cos/sin/log, which the storage rounding
# almost always absorbs.


def _as_i64(x: int) -> int:
    x &= 0xFFFFFFFFFFFFFFFF
    return x - (1 << 64) if x >= (1 << 63) else x


def _lsr(z, s: int):
    """Logical right shift of int64 values (two's-complement bit pattern)."""
    import torch

    return (z >> s) & torch.tensor((1 << (64 - s)) - 1, dtype=torch.int64, device=z.device)


def normal_device(seed: int, n: int, device, chunk: int = 1 << 24):
    import torch

    m = (n + 1) // 2
    out = torch.empty(2 * m, dtype=torch.float64, device=device)
    g, m1, m2 = _as_i64(0x9E3779B97F4A7C15), _as_i64(0xBF58476D1CE4E5B9), _as_i64(0x94D049BB133111EB)
    s0 = _as_i64(seed)
    for lo in range(0, 2 * m, chunk):
        hi = min(2 * m, lo + chunk)
        z = torch.arange(lo + 1, hi + 1, dtype=torch.int64, device=device) * g + s0
        z = (z ^ _lsr(z, 30)) * m1
        z = (z ^ _lsr(z, 27)) * m2
        z = z ^ _lsr(z, 31)
        u = _lsr(z, 11).to(torch.float64) * (1.0 / 9007199254740992.0)
        r = torch.sqrt(-2.0 * torch.log1p(-u[0::2]))
        t = 2.0 * torch.pi * u[1::2]
        out[lo:hi:2] = r * torch.cos(t)
        out[lo + 1 : hi : 2] = r * torch.sin(t)
    return out[:n]


def make_qkvdo_device(B, T, Hq, Hkv, D, dtype: str, seed: int, device, layer: int = 0,
                      with_do: bool = True):
    """``make_qkvdo`` generated directly on ``device``."""
    import torch

    tdt = {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]

    def one(shape, tid):
        n = int(np.prod(shape))
        x = normal_device(mix_seed(seed, layer, tid), n, device)
        return x.to(torch.float32).to(tdt).reshape(shape)

    out = {"q": one((B, Hq, T, D), TENSOR_IDS["q"]), "k": one((B, Hkv, T, D), TENSOR_IDS["k"]),
           "v": one((B, Hkv, T, D), TENSOR_IDS["v"])}
    if with_do:
        out["do"] = one((B, Hq, T, D), TENSOR_IDS["do"])
    return out
