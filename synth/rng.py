"""Counter-based SplitMix64 random numbers, vectorised with numpy.

SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014; the 64-bit finaliser constants as published by
Vigna) is used here in counter mode: draw number ``i`` of stream ``s`` under
seed ``seed`` is the SplitMix64 finaliser applied to
``key(seed, s) + (i + 1) * 0x9E3779B97F4A7C15`` (mod 2**64).  Every draw is a
pure function of ``(seed, stream, i)``, so the inputs are identical on every
machine and numpy version, and any subset of draws can be regenerated without
producing the ones before it.

This module holds no sparse-matrix arithmetic; it only produces numbers.
"""
from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_TWO_M53 = 1.0 / 9007199254740992.0  # 2**-53


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output finaliser, in place on a uint64 array (wrapping arithmetic)."""
    t = np.empty_like(z)
    np.right_shift(z, np.uint64(30), out=t)
    z ^= t
    z *= _M1
    np.right_shift(z, np.uint64(27), out=t)
    z ^= t
    z *= _M2
    np.right_shift(z, np.uint64(31), out=t)
    z ^= t
    return z


_CHUNK = 1 << 20


def stream_key(seed: int, stream: int) -> np.uint64:
    """Key of one named stream: the finaliser of a fixed combination of both ids."""
    base = (int(seed) * 0x100000001B3 + int(stream) * 0x9E3779B97F4A7C15 + 0x243F6A8885A308D3)
    return _mix(np.array([base & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0]


def raw_u64(seed: int, stream: int, count: int, offset: int = 0) -> np.ndarray:
    """Draws ``offset .. offset+count-1`` of a stream as uint64."""
    key = stream_key(seed, stream)
    out = np.empty(count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        for s0 in range(0, count, _CHUNK):
            s1 = min(count, s0 + _CHUNK)
            z = out[s0:s1]
            z[:] = np.arange(offset + s0 + 1, offset + s1 + 1, dtype=np.uint64)
            z *= _GOLDEN
            z += key
            _mix(z)
    return out


def raw_at(seed: int, stream: int, counters: np.ndarray) -> np.ndarray:
    """Draws at arbitrary (non-negative integer) counters of a stream."""
    key = stream_key(seed, stream)
    with np.errstate(over="ignore"):
        z = (np.asarray(counters, dtype=np.uint64) + np.uint64(1)) * _GOLDEN
        z += key
    return _mix(z)


def to_unit(z: np.ndarray) -> np.ndarray:
    """uint64 -> float64 uniform on [0, 1) using the top 53 bits."""
    return (z >> np.uint64(11)).astype(np.float64) * _TWO_M53


def to_unit_open0(z: np.ndarray) -> np.ndarray:
    """uint64 -> float64 uniform on (0, 1] (safe for log)."""
    return ((z >> np.uint64(11)).astype(np.float64) + 1.0) * _TWO_M53


def uniform(seed: int, stream: int, count: int, lo: float = 0.0, hi: float = 1.0,
            offset: int = 0) -> np.ndarray:
    return lo + (hi - lo) * to_unit(raw_u64(seed, stream, count, offset))


def normal(seed: int, stream: int, count: int) -> np.ndarray:
    """Standard normals by the Box-Muller transform over two sub-streams."""
    out = np.empty(count, dtype=np.float64)
    for s0 in range(0, count, _CHUNK):
        c = min(count, s0 + _CHUNK) - s0
        u1 = to_unit_open0(raw_u64(seed, stream * 2 + 1_000_001, c, s0))
        u2 = to_unit(raw_u64(seed, stream * 2 + 1_000_002, c, s0))
        np.log(u1, out=u1)
        u1 *= -2.0
        np.sqrt(u1, out=u1)
        u2 *= 2.0 * np.pi
        np.cos(u2, out=u2)
        np.multiply(u1, u2, out=out[s0:s0 + c])
    return out


def exponential(seed: int, stream: int, count: int) -> np.ndarray:
    """Exp(1) draws as -log(U), U uniform on (0, 1]."""
    return -np.log(to_unit_open0(raw_u64(seed, stream, count)))


def integers(seed: int, stream: int, count: int, lo: int, hi: int) -> np.ndarray:
    """Integers uniform on [lo, hi] (inclusive) by scaling the 53-bit uniform."""
    span = hi - lo + 1
    return lo + np.floor(to_unit(raw_u64(seed, stream, count)) * span).astype(np.int64)
