"""Seeded synthetic GEMM operands, shared by the CUDA path's tests/bench and the oracle's.

This module only draws numbers.  It holds none of the GEMM arithmetic, so both
sides of every parity test can take their inputs from here without sharing any
part of the computation under test.

Random stream
-------------
Counter-based SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014; the finaliser constants are the published
ones).  Element ``i`` of stream ``(seed, tag)`` is ``mix64(base + (i + 1) * GAMMA)``
with ``base = mix64(seed * 2**32 + tag)``.  Being counter-based, any sub-range
can be regenerated alone and the output does not depend on chunking.

Distributions (all exact in the stored type)
--------------------------------------------
* ``uniform``: the top 24 bits ``u`` of a draw give ``u * 2**-23 - 1``, a value
  in [-1, 1) that is a multiple of 2**-23 and therefore exact in float32.
* ``normal(sigma)``: Box-Muller in float64 from two draws (indices 2i, 2i+1),
  scaled by sigma, rounded to float32 (round to nearest even).
* ``smallint(lo, hi)``: integers in [lo, hi], exact in float32 and bfloat16.
* BF16 operands are float32 values rounded to bfloat16 by round-to-nearest-even
  and returned as raw uint16 bit patterns.

Layout
------
Row-major ``rows x cols`` with leading dimension ``ld >= cols``; element (r, c)
takes logical draw index ``r * cols + c`` so padding never shifts the values.
Padding elements (columns ``cols .. ld-1``) are NaN for float32 (a kernel that
reads them poisons its output) and 0x7FC0 (a bfloat16 NaN) for bfloat16.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK64 = (1 << 64) - 1

# Stream tags: operand A and operand B of one configuration never share draws.
TAG_A = 1
TAG_B = 2

_CHUNK = 1 << 20


def _mix64_array(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser on a uint64 array, in place (wrap-around arithmetic)."""
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


def _mix64_int(x: int) -> int:
    z = x & _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def draws(seed: int, tag: int, start: int, count: int) -> np.ndarray:
    """Raw 64-bit draws ``start .. start+count-1`` of stream (seed, tag)."""
    base = np.uint64(_mix64_int((seed << 32) + tag))
    z = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z *= _GAMMA
        z += base
    return _mix64_array(z)


def _fill_logical(n: int, fn) -> np.ndarray:
    """Evaluate ``fn(start, count)`` chunk by chunk into one float32 vector.

    Chunks are independent (the stream is counter-based), so they run on a
    thread pool; numpy releases the GIL inside each operation."""
    out = np.empty(n, dtype=np.float32)
    starts = list(range(0, n, _CHUNK))

    def one(s):
        c = min(_CHUNK, n - s)
        out[s:s + c] = fn(s, c)

    if len(starts) <= 1:
        for s in starts:
            one(s)
    else:
        workers = min(len(starts), os.cpu_count() or 1, 32)
        with ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(one, starts))
    return out


def uniform_values(seed: int, tag: int, n: int) -> np.ndarray:
    def chunk(s, c):
        u = (draws(seed, tag, s, c) >> np.uint64(40)).astype(np.float64)
        return (u * 2.0 ** -23 - 1.0).astype(np.float32)
    return _fill_logical(n, chunk)


def normal_values(seed: int, tag: int, n: int, sigma: float) -> np.ndarray:
    def chunk(s, c):
        z = draws(seed, tag, 2 * s, 2 * c)
        u1 = ((z[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
        u2 = (z[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        g = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
        return (sigma * g).astype(np.float32)
    return _fill_logical(n, chunk)


def smallint_values(seed: int, tag: int, n: int, lo: int = -2, hi: int = 2) -> np.ndarray:
    span = np.uint64(hi - lo + 1)

    def chunk(s, c):
        z = draws(seed, tag, s, c) >> np.uint64(32)
        return ((z % span).astype(np.int64) + lo).astype(np.float32)
    return _fill_logical(n, chunk)


def _place(values: np.ndarray, rows: int, cols: int, ld: int, pad) -> np.ndarray:
    if ld < cols:
        raise ValueError(f"leading dimension {ld} < cols {cols}")
    out = np.full((rows, ld), pad, dtype=values.dtype)
    out[:, :cols] = values.reshape(rows, cols)
    return out


def matrix_f32(kind: str, rows: int, cols: int, seed: int, tag: int,
               ld: int | None = None, sigma: float = 1.0) -> np.ndarray:
    """A ``rows x ld`` float32 array; columns ``>= cols`` are NaN padding.

    ``kind``: 'uniform' | 'normal' | 'smallint' | 'ones' | 'zeros' | 'identity' | 'page4a' | 'page4b'.
    The 'page4a'/'page4b' patterns are the day-74 program's own inputs
    (pipelined_gemm.cu, ``main``): a[i] = (i % 97) * 0.01f and
    b[i] = (i % 53) * 0.02f - 0.5f over the flat logical index.
    """
    ld = cols if ld is None else ld
    n = rows * cols
    if kind == "uniform":
        v = uniform_values(seed, tag, n)
    elif kind == "normal":
        v = normal_values(seed, tag, n, sigma)
    elif kind == "smallint":
        v = smallint_values(seed, tag, n)
    elif kind == "ones":
        v = np.ones(n, dtype=np.float32)
    elif kind == "zeros":
        v = np.zeros(n, dtype=np.float32)
    elif kind == "identity":
        v = np.eye(rows, cols, dtype=np.float32).reshape(-1)
    elif kind == "page4a":
        i = np.arange(n, dtype=np.int64)
        v = (i % 97).astype(np.float32) * np.float32(0.01)
    elif kind == "page4b":
        i = np.arange(n, dtype=np.int64)
        v = (i % 53).astype(np.float32) * np.float32(0.02) - np.float32(0.5)
    else:
        raise ValueError(f"unknown kind {kind!r}")
    return _place(v.astype(np.float32), rows, cols, ld, np.float32(np.nan))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); return uint16 bits.

    NaN inputs map to the quiet bfloat16 NaN 0x7FC0.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    out = rounded.astype(np.uint16)
    out[np.isnan(x)] = np.uint16(0x7FC0)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 exactly."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def matrix_bf16(kind: str, rows: int, cols: int, seed: int, tag: int,
                ld: int | None = None, sigma: float = 1.0) -> np.ndarray:
    """A ``rows x ld`` uint16 array of bfloat16 bits (padding = bf16 NaN)."""
    f = matrix_f32(kind, rows, cols, seed, tag, ld=ld, sigma=sigma)
    return f32_to_bf16_bits(f)


# The five workloads the library is specified and measured on.  Each entry:
# (M, N, K, lda, A/B distribution, sigma, seed).
WORKLOADS = {
    "f32_256": dict(M=256, N=256, K=256, lda=256, kind="uniform", sigma=1.0, seed=0),
    "f32_1024": dict(M=1024, N=1024, K=1024, lda=1024, kind="uniform", sigma=1.0, seed=1),
    "f32_4096": dict(M=4096, N=4096, K=4096, lda=4096, kind="uniform", sigma=1.0, seed=2),
    "f32_ragged": dict(M=3000, N=5000, K=1000, lda=1003, kind="normal", sigma=1.0, seed=3),
    "bf16_8192": dict(M=8192, N=8192, K=8192, lda=8192, kind="normal", sigma=0.5, seed=4),
    # The latency-bound shape of "A study on CUDA async memcpy" ("Real world
    # example": M = N = 32, K = 65536, one block); seed 5 is this library's choice.
    "f32_tallk": dict(M=32, N=32, K=65536, lda=65536, kind="uniform", sigma=1.0, seed=5),
}


def workload_operands(name: str, lda: int | None = None):
    """(A, B) host arrays for a named workload; BF16 workloads return uint16 bits."""
    w = WORKLOADS[name]
    lda = w["lda"] if lda is None else lda
    if name.startswith("bf16"):
        a = matrix_bf16(w["kind"], w["M"], w["K"], w["seed"], TAG_A, ld=lda, sigma=w["sigma"])
        b = matrix_bf16(w["kind"], w["K"], w["N"], w["seed"], TAG_B, sigma=w["sigma"])
    else:
        a = matrix_f32(w["kind"], w["M"], w["K"], w["seed"], TAG_A, ld=lda, sigma=w["sigma"])
        b = matrix_f32(w["kind"], w["K"], w["N"], w["seed"], TAG_B, sigma=w["sigma"])
    return a, b
