"""Seeded synthetic inputs shared by the tests and the benchmark.

This module holds no arithmetic of the method: it only draws numbers.  The
generator is splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014): a 64-bit Weyl sequence with increment
0x9E3779B97F4A7C15 passed through the published mixing function.  Normal
variates come from the Box-Muller transform in fp64, rounded once to fp32.

A (seed, stream) pair names an independent sequence: its start state is
seed * 0x9E3779B97F4A7C15 + stream * 0xD1B54A32D192ED03 (mod 2^64), and the
i-th output is mix(start + (i + 1) * 0x9E3779B97F4A7C15).  Element i of a
normal array uses outputs 2*(i//2) and 2*(i//2)+1 (cos branch for even i,
sin branch for odd i).

Two implementations of the same definition are provided: numpy (the one the
parity tests use on both sides) and torch on any device (used to fill large
benchmark caches quickly; its transcendental functions may differ from
numpy's in the last fp64 bit, so its fp32 outputs are not promised to be
bit-identical to the numpy ones).
"""
from __future__ import annotations

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
STREAM_MUL = 0xD1B54A32D192ED03
M1 = 0xBF58476D1CE4E5B9
M2 = 0x94D049BB133111EB
_MASK = (1 << 64) - 1


def _start(seed: int, stream: int) -> int:
    return (seed * GOLDEN + stream * STREAM_MUL) & _MASK


def _mix_np(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(M1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(M2)
    return z ^ (z >> np.uint64(31))


def raw_u64(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """Outputs offset .. offset+n-1 of the (seed, stream) sequence."""
    with np.errstate(over="ignore"):
        i = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        z = np.uint64(_start(seed, stream)) + i * np.uint64(GOLDEN)
        return _mix_np(z)


def uniform01(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """Uniforms in (0, 1] from the top 53 bits, fp64."""
    x = raw_u64(seed, stream, n, offset)
    return ((x >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def normal(seed: int, stream: int, n: int, sigma: float = 1.0) -> np.ndarray:
    """n N(0, sigma^2) variates as fp32 (Box-Muller in fp64)."""
    pairs = (n + 1) // 2
    u = uniform01(seed, stream, 2 * pairs)
    u1, u2 = u[0::2], u[1::2]
    rad = np.sqrt(-2.0 * np.log(u1))
    out = np.empty(2 * pairs, dtype=np.float64)
    out[0::2] = rad * np.cos(2.0 * np.pi * u2)
    out[1::2] = rad * np.sin(2.0 * np.pi * u2)
    return (out[:n] * sigma).astype(np.float32)


def randint(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers uniform in [lo, hi] (inclusive)."""
    u = uniform01(seed, stream, n)  # (0, 1]
    span = hi - lo + 1
    v = np.floor((1.0 - u) * span).astype(np.int64)  # [0, span)
    return (lo + np.minimum(v, span - 1)).astype(np.int64)


# Stream ids: one per (layer, tensor) so that every tensor is independent.
def stream_id(kind: str, layer: int = 0, extra: int = 0) -> int:
    kinds = {"k": 1, "v": 2, "q": 3, "len": 4, "knew": 5, "vnew": 6, "misc": 7}
    return (kinds[kind] << 40) | (layer << 20) | extra


def normal_torch(seed: int, stream: int, n: int, sigma: float = 1.0, device="cpu"):
    """Same definition as normal(), computed with torch on `device`."""
    import torch

    pairs = (n + 1) // 2
    i = torch.arange(1, 2 * pairs + 1, dtype=torch.int64, device=device)

    def s64(v: int) -> int:  # reinterpret an unsigned 64-bit constant as int64
        v &= _MASK
        return v - (1 << 64) if v >= (1 << 63) else v

    def shr(x, k):  # logical right shift on int64
        return (x >> k) & ((1 << (64 - k)) - 1)

    z = i * s64(GOLDEN) + s64(_start(seed, stream))
    z = (z ^ shr(z, 30)) * s64(M1)
    z = (z ^ shr(z, 27)) * s64(M2)
    z = z ^ shr(z, 31)
    u = (shr(z, 11).to(torch.float64) + 1.0) * (2.0 ** -53)
    u1, u2 = u[0::2], u[1::2]
    rad = torch.sqrt(-2.0 * torch.log(u1))
    out = torch.empty(2 * pairs, dtype=torch.float64, device=device)
    out[0::2] = rad * torch.cos(2.0 * np.pi * u2)
    out[1::2] = rad * torch.sin(2.0 * np.pi * u2)
    return (out[:n] * sigma).to(torch.float32)
