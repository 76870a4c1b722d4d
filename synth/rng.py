"""Counter-based random numbers for the seeded synthetic workloads.

Every value is a pure function of (key, counter), so any element of any tensor
can be regenerated on its own (the oracle's sampled checks rely on this) and the
same numbers come out on x86 and aarch64.

* splitmix64 -- Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators" (OOPSLA 2014): the output mix of state ``key + (i+1)*gamma``.
* Box-Muller -- Box & Muller (1958): two uniforms (0,1) -> two N(0,1).
* bf16 rounding -- round-to-nearest-even of the fp64 value to an 8-bit
  significand, then the top 16 bits of the (exact) fp32 encoding.

This module holds input generation only; none of the attention arithmetic.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_S30, _S27, _S31, _S11 = (np.uint64(s) for s in (30, 27, 31, 11))
_MASK64 = (1 << 64) - 1


def _mix_inplace(z: np.ndarray) -> np.ndarray:
    z ^= z >> _S30
    z *= _M1
    z ^= z >> _S27
    z *= _M2
    z ^= z >> _S31
    return z


def splitmix64(key: int, counters: np.ndarray) -> np.ndarray:
    """64-bit outputs for the given counters of the stream ``key``."""
    c = np.asarray(counters, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (c + np.uint64(1)) * _GAMMA
        z += np.uint64(key & _MASK64)
        return _mix_inplace(z)


def splitmix64_scalar(key: int, counter: int) -> int:
    z = (key + (counter + 1) * 0x9E3779B97F4A7C15) & _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, *tags: int) -> int:
    """Derive an independent stream key from a seed and integer tags."""
    k = splitmix64_scalar(seed & _MASK64, 0x5EED)
    for t in tags:
        k = splitmix64_scalar(k, t & _MASK64)
    return k


def uniform01(key: int, counters: np.ndarray) -> np.ndarray:
    """Uniform doubles in the open interval (0, 1): (top 53 bits + 0.5) / 2^53."""
    z = splitmix64(key, counters)
    return ((z >> _S11).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)


def uniform_int(key: int, counter: int, lo: int, hi: int) -> int:
    """One integer uniform on [lo, hi] (inclusive) by rejection (no modulo bias)."""
    span = hi - lo + 1
    limit = (1 << 64) - ((1 << 64) % span)
    c = counter
    while True:
        z = splitmix64_scalar(key, c)
        if z < limit:
            return lo + z % span
        c += 1 << 40  # rejected draws move to a far-away counter range


def uniform_real(key: int, counter: int) -> float:
    z = splitmix64_scalar(key, counter)
    return ((z >> 11) + 0.5) / 9007199254740992.0


def normal(key: int, start: int, n: int) -> np.ndarray:
    """Standard normals with indices start..start+n-1 of stream ``key``.

    Index j uses the uniform pair (2*(j//2), 2*(j//2)+1); even j takes the
    cosine branch, odd j the sine branch.
    """
    j = np.arange(start, start + n, dtype=np.uint64)
    return normal_at(key, j)


def normal_at(key: int, idx: np.ndarray) -> np.ndarray:
    """Standard normals at arbitrary (uint64) indices of stream ``key``."""
    idx = np.asarray(idx, dtype=np.uint64)
    pair = idx >> np.uint64(1)
    u1 = uniform01(key, pair * np.uint64(2))
    u2 = uniform01(key, pair * np.uint64(2) + np.uint64(1))
    r = np.sqrt(-2.0 * np.log(u1))
    theta = (2.0 * np.pi) * u2
    odd = (idx & np.uint64(1)).astype(bool)
    return np.where(odd, r * np.sin(theta), r * np.cos(theta))


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 bit patterns (uint16), one round-to-nearest-even step.

    The value is rounded once to an 8-bit significand (np.rint is
    half-to-even), which is then exact in fp32; its top 16 bits are the bf16.
    Values are N(0,1)-sized, far from the bf16 overflow and subnormal ranges.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                       # x = m * 2^e, 0.5 <= |m| < 1
    r = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
    f32 = r.astype(np.float32)               # exact: 8 significant bits
    return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def parallel_fill(n_items: int, fn, workers: int | None = None, min_chunk: int = 1):
    """Run fn(lo, hi) over [0, n_items) in chunks on a thread pool.

    numpy releases the GIL in its vectorised kernels, so threads scale; no
    process is forked (safe after CUDA is initialised).
    """
    if n_items <= 0:
        return
    workers = workers or min(32, os.cpu_count() or 1)
    n_chunks = max(1, min(workers * 4, n_items // max(1, min_chunk)))
    bounds = np.linspace(0, n_items, n_chunks + 1).astype(np.int64)
    if n_chunks == 1:
        fn(0, n_items)
        return
    with _cf.ThreadPoolExecutor(max_workers=workers) as ex:
        futs = [ex.submit(fn, int(bounds[i]), int(bounds[i + 1]))
                for i in range(n_chunks) if bounds[i + 1] > bounds[i]]
        for f in futs:
            f.result()
