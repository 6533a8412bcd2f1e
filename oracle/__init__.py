"""CPU GEMM oracle: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The CUDA product path never reaches
it, and it shares no code with the CUDA path (the only common module is the
seeded input generator, which holds no GEMM arithmetic).

Functions (thin ctypes wrappers over ``gemm_oracle.c``; see that file for the
definitions and the passages they follow):

* ``gemm_f64(A, B, M, N, K)``: the plain definition, float64 accumulation.
* ``gemm_fmaf_chain(A, B, M, N, K)``: float32 fused-multiply-add chain per
  element, k ascending from +0 (the kernels' arithmetic, written out).
* ``gemm_bf16_f64(A_bits, B_bits, M, N, K)``: bfloat16 operands widened
  exactly, float64 accumulation.

Operands are numpy arrays, row-major, with leading dimension = the array's
second extent (so padded arrays pass their padding through untouched).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libgemm_oracle.so")
_lock = threading.Lock()
_lib = None


GCC_FLAGS = ["-O2", "-std=c99", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def compile_source(src: str, out: str) -> str:
    """gcc one oracle source file into a shared library at ``out``."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *GCC_FLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def _fresh() -> bool:
    return os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, OpenMP, no fast-math); one build
    at a time per tree."""
    if not force and _fresh():
        return _LIB_PATH
    import fcntl
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    with open(_LIB_PATH + ".lock", "w") as f:
        fcntl.flock(f, fcntl.LOCK_EX)
        try:
            if force or not _fresh():
                compile_source(_SRC, _LIB_PATH)
        finally:
            fcntl.flock(f, fcntl.LOCK_UN)
    return _LIB_PATH


def load_variant(path: str):
    """Bind a separately compiled build of gemm_oracle.c (used by the tests
    that plant mistakes in the oracle to show that the pins catch them)."""
    return _bind(ctypes.CDLL(path))


def _bind(lib):
    L, P = ctypes.c_long, ctypes.c_void_p
    for name in ("oracle_gemm_f64", "oracle_gemm_fmaf_chain", "oracle_gemm_bf16_f64"):
        fn = getattr(lib, name)
        fn.argtypes = [L, L, L, P, L, P, L, P, L]
        fn.restype = None
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    lib.oracle_set_num_threads.restype = None
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _check(x: np.ndarray, dtype, rows: int, cols: int, name: str) -> np.ndarray:
    if x.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {x.dtype}")
    if x.ndim != 2 or x.shape[0] < rows or x.shape[1] < cols:
        raise ValueError(f"{name}: shape {x.shape} too small for {rows}x{cols}")
    if x.strides[1] != x.itemsize:
        raise ValueError(f"{name}: rows must be contiguous")
    return x


def _ld(x: np.ndarray) -> int:
    return x.strides[0] // x.itemsize


def _ptr(x: np.ndarray) -> int:
    return x.ctypes.data


def gemm_f64(A: np.ndarray, B: np.ndarray, M: int, N: int, K: int, lib=None) -> np.ndarray:
    """float64 M x N result of A[:M,:K] @ B[:K,:N] (float32 operands)."""
    _check(A, np.float32, M, K, "A")
    _check(B, np.float32, K, N, "B")
    C = np.empty((M, N), dtype=np.float64)
    if M and N:
        (lib or _load()).oracle_gemm_f64(M, N, K, _ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(C), N)
    return C


def gemm_fmaf_chain(A: np.ndarray, B: np.ndarray, M: int, N: int, K: int, lib=None) -> np.ndarray:
    """float32 M x N result, one fmaf chain per element, k ascending from +0."""
    _check(A, np.float32, M, K, "A")
    _check(B, np.float32, K, N, "B")
    C = np.empty((M, N), dtype=np.float32)
    if M and N:
        (lib or _load()).oracle_gemm_fmaf_chain(M, N, K, _ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(C), N)
    return C


def gemm_bf16_f64(A: np.ndarray, B: np.ndarray, M: int, N: int, K: int, lib=None) -> np.ndarray:
    """float64 M x N result for bfloat16 operands given as uint16 bit arrays."""
    _check(A, np.uint16, M, K, "A")
    _check(B, np.uint16, K, N, "B")
    C = np.empty((M, N), dtype=np.float64)
    if M and N:
        (lib or _load()).oracle_gemm_bf16_f64(M, N, K, _ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(C), N)
    return C


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))
