"""Counter-based random numbers for the synthetic workloads.

Every random value is a pure function of (seed, stream, index), so a workload
is identical on every machine and no state is carried between calls.  The mixer
is SplitMix64 (G. L. Steele, D. Lea, C. H. Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014): a 64-bit counter advanced by the golden-ratio
increment 0x9E3779B97F4A7C15, then finalised by two xor-shift-multiply rounds.

    key(seed, stream) = mix(seed * 2**20 + stream)
    bits(seed, stream, i) = mix(key + (i + 1) * 0x9E3779B97F4A7C15)

Uniforms take the top 53 bits (u = bits >> 11, times 2**-53, so u in [0, 1)).
Normals use the Box-Muller transform on the uniform pair (2i, 2i + 1).
Nothing here knows about sparse matrices or solvers.
"""
from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser, applied elementwise to a uint64 array."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int) -> np.uint64:
    base = np.array([(int(seed) << 20) + int(stream)], dtype=np.uint64)
    return _mix(base)[0]


def bits(seed: int, stream: int, count: int, offset: int = 0) -> np.ndarray:
    """uint64 draws number offset .. offset + count - 1 of (seed, stream)."""
    key = stream_key(seed, stream)
    idx = np.arange(offset + 1, offset + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + idx * _GOLDEN)


def uniform(seed: int, stream: int, count: int, offset: int = 0) -> np.ndarray:
    """float64 uniforms in [0, 1)."""
    b = bits(seed, stream, count, offset)
    return (b >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def uniform_pm1(seed: int, stream: int, count: int, offset: int = 0) -> np.ndarray:
    """float64 uniforms in [-1, 1)."""
    return 2.0 * uniform(seed, stream, count, offset) - 1.0


def normal(seed: int, stream: int, count: int, offset: int = 0) -> np.ndarray:
    """Standard normals by Box-Muller on uniform pairs (2i, 2i + 1)."""
    u = uniform(seed, stream, 2 * count, 2 * offset)
    u1 = 1.0 - u[0::2]  # in (0, 1], so the log is finite
    u2 = u[1::2]
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    """A seeded random permutation of 0..n-1 (stable argsort of random keys)."""
    return np.argsort(bits(seed, stream, n), kind="stable").astype(np.int64)
