"""Seeded synthetic inputs for the FP32 matrix product C[M x K] = A[M x N] . B[N x K].

This module only draws numbers. It holds none of the product's arithmetic, so the
CUDA path and the CPU oracle can both be fed from it without sharing any code that
computes a result.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014), used counter-style. Draw number i of stream ``seed`` is the
i-th output of SplitMix64 started from state ``seed``:

    state_i = seed + (i + 1) * 0x9E3779B97F4A7C15          (mod 2^64)
    z = (state_i ^ (state_i >> 30)) * 0xBF58476D1CE4E5B9
    z = (z ^ (z >> 27)) * 0x94D049BB133111EB
    draw_i = z ^ (z >> 31)

One draw per element in row-major order, A first and then B (two draws per element for
the normal distribution). Distributions:

* ``"uniform"``: uniform on [-1, 1) as ((d >> 40) * 2^-24) * 2 - 1. Every value is an
  exact float32 (a 24-bit integer scaled by 2^-23).
* ``"uniform01"``: uniform on [0, 1) as (d >> 40) * 2^-24, every value an exact float32;
  all entries of one sign, the case where accumulation error does not cancel.
* ``"int4"`` / ``"int8"`` / ``"int<a>"``: integers uniform on [-a, a] inclusive,
  (d mod (2a + 1)) - a.
* ``"normal"``: N(0, 1) by Box-Muller in float64 from draws (2i, 2i+1), rounded to
  float32.

The workloads these feed are the problem statement's shapes (1 <= M, N, K <= 8192 and the
performance shape M=8192, N=6144, K=4096 of "LeetGPU | 02_Matrix_Multiplication",
section "Constraints").
"""

from __future__ import annotations

import os

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 20
_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        from concurrent.futures import ThreadPoolExecutor
        _POOL = ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1)))
    return _POOL


def _mix_into(out: np.ndarray, seed: int, first: int) -> None:
    """out[j] = draw number (first + j) of the SplitMix64 stream started at seed."""
    n = out.shape[0]
    out[:] = np.arange(first + 1, first + n + 1, dtype=np.uint64)
    tmp = np.empty_like(out)
    with np.errstate(over="ignore"):
        np.multiply(out, _GAMMA, out=out)
        np.add(out, np.uint64(seed & 0xFFFFFFFFFFFFFFFF), out=out)
        np.right_shift(out, np.uint64(30), out=tmp)
        np.bitwise_xor(out, tmp, out=out)
        np.multiply(out, _MIX1, out=out)
        np.right_shift(out, np.uint64(27), out=tmp)
        np.bitwise_xor(out, tmp, out=out)
        np.multiply(out, _MIX2, out=out)
        np.right_shift(out, np.uint64(31), out=tmp)
        np.bitwise_xor(out, tmp, out=out)


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of the SplitMix64 stream started at ``seed``."""
    out = np.empty(count, dtype=np.uint64)
    _mix_into(out, seed, start)
    return out


def _fill_chunk(out: np.ndarray, seed: int, first: int, dist: str) -> None:
    n = out.shape[0]
    if dist == "uniform":
        d = np.empty(n, dtype=np.uint64)
        _mix_into(d, seed, first)
        np.right_shift(d, np.uint64(40), out=d)
        # (d >> 40) * 2^-24 * 2 - 1, exact in float32 (24-bit integer times 2^-23, minus 1)
        u = d.astype(np.float32)
        np.multiply(u, np.float32(2.0 ** -23), out=u)
        np.subtract(u, np.float32(1.0), out=out)
    elif dist == "uniform01":
        d = np.empty(n, dtype=np.uint64)
        _mix_into(d, seed, first)
        np.right_shift(d, np.uint64(40), out=d)
        # (d >> 40) * 2^-24: a 24-bit integer scaled by a power of two, exact in float32
        np.multiply(d.astype(np.float32), np.float32(2.0 ** -24), out=out)
    elif dist.startswith("int"):
        a = int(dist[3:])
        d = np.empty(n, dtype=np.uint64)
        _mix_into(d, seed, first)
        np.remainder(d, np.uint64(2 * a + 1), out=d)
        out[:] = d.astype(np.int64) - a
    elif dist == "normal":
        d = np.empty(2 * n, dtype=np.uint64)
        _mix_into(d, seed, 2 * first)
        u1 = ((d[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
        u2 = (d[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        out[:] = (np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)).astype(np.float32)
    else:
        raise ValueError(f"unknown distribution {dist!r}")


def _draws_to_values(seed: int, start: int, count: int, dist: str) -> np.ndarray:
    if dist not in ("uniform", "uniform01", "normal") and not (dist.startswith("int") and dist[3:].isdigit()):
        raise ValueError(f"unknown distribution {dist!r}")
    out = np.empty(count, dtype=np.float32)
    futs = [_pool().submit(_fill_chunk, out[lo:min(count, lo + _CHUNK)], seed, start + lo, dist)
            for lo in range(0, count, _CHUNK)]
    for f in futs:
        f.result()
    return out


def make_inputs(M: int, N: int, K: int, seed: int, dist: str = "uniform"):
    """Returns (A, B): A is M x N and B is N x K, C-contiguous float32 arrays.

    A takes draws 0 .. M*N-1 and B takes the draws after it, so A is the same whatever K is.
    """
    a = _draws_to_values(seed, 0, M * N, dist).reshape(M, N)
    b = _draws_to_values(seed, M * N, N * K, dist).reshape(N, K)
    return a, b


def make_permutation(n: int, seed: int) -> np.ndarray:
    """A permutation of 0..n-1 from SplitMix64 draws (Fisher-Yates, high-to-low)."""
    d = splitmix64(seed ^ 0x5EED, 0, max(n, 1))
    p = np.arange(n, dtype=np.int64)
    for i in range(n - 1, 0, -1):
        j = int(d[i] % np.uint64(i + 1))
        p[i], p[j] = p[j], p[i]
    return p


def sample_indices(M: int, K: int, count: int, seed: int):
    """``count`` output coordinates (row, col) drawn from SplitMix64, always including the
    four corners, for spot checks of outputs too large to compute in full on the CPU."""
    d = splitmix64(seed ^ 0xC0FFEE, 0, 2 * count)
    rows = (d[0::2] % np.uint64(M)).astype(np.int64)
    cols = (d[1::2] % np.uint64(K)).astype(np.int64)
    corners_r = np.array([0, 0, M - 1, M - 1], dtype=np.int64)
    corners_c = np.array([0, K - 1, 0, K - 1], dtype=np.int64)
    return np.concatenate([corners_r, rows]), np.concatenate([corners_c, cols])
