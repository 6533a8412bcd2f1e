"""Helpers shared by the GPU parity tests: move seeded host operands to the
device (keeping their padding), run the library through its C ABI binding,
and evaluate the oracle on the same host arrays (whole or on sampled rows)."""
from __future__ import annotations

import numpy as np

import oracle
from async_copy_pipelined_gb300 import inputs

# (fill, stages, tile) combinations of the FP32 kernel family.
F32_VARIANTS = [("sync", 1, 32), ("sync", 1, 64), ("sync", 1, 128)]
F32_VARIANTS += [(f, s, t) for f in ("cpasync", "tma", "cpasync_mbar", "cpasync_ws") for s in (2, 3, 4, 5, 6)
                 for t in (32, 64, 128)]


def to_device(x: np.ndarray, cols: int):
    """Copy a padded host matrix (rows x ld) to the GPU; return the logical
    rows x cols view whose row stride is ld."""
    import torch
    if x.dtype == np.uint16:
        t = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(x))
    return t.cuda()[:, :cols]


def run_f32(A: np.ndarray, B: np.ndarray, M: int, N: int, K: int, fill: str, stages: int, tile: int,
            ldc: int | None = None, sentinel: float = 12345.0):
    """Run gemm_f32 and return (C logical M x N, full C buffer M x ldc) on the host."""
    import torch
    import async_copy_pipelined_gb300 as pg
    Ad = to_device(A, K)
    Bd = to_device(B, N)
    ldc = N if ldc is None else ldc
    Cbuf = torch.full((M, max(ldc, 1)), sentinel, dtype=torch.float32, device="cuda")
    C = Cbuf[:, :N]
    pg.gemm_f32(Ad, Bd, C, fill=fill, stages=0 if fill == "sync" else stages, block_tile=tile)
    st, detail = pg.device_status()
    assert st == 0, f"device status {st} detail {detail:#x}"
    torch.cuda.synchronize()
    full = Cbuf.cpu().numpy()
    return full[:, :N].copy(), full


def run_bf16(A: np.ndarray, B: np.ndarray, M: int, N: int, K: int, stages: int = 0, ldc: int | None = None,
             sentinel: float = 12345.0, fill: str = "tma", block_m: int = 0):
    import torch
    import async_copy_pipelined_gb300 as pg
    Ad = to_device(A, K)
    Bd = to_device(B, N)
    ldc = N if ldc is None else ldc
    Cbuf = torch.full((M, max(ldc, 1)), sentinel, dtype=torch.float32, device="cuda")
    C = Cbuf[:, :N]
    pg.gemm_bf16(Ad, Bd, C, fill=fill, stages=stages, block_m=block_m)
    st, detail = pg.device_status()
    assert st == 0, f"device status {st} detail {detail:#x}"
    torch.cuda.synchronize()
    full = Cbuf.cpu().numpy()
    return full[:, :N].copy(), full


def sample_rows(M: int, count: int, seed: int, tiles=(64, 128)) -> np.ndarray:
    """Edge rows (first/last of every tile boundary near the ends) plus random rows."""
    rows = {0, 1, M - 1, M - 2}
    for t in tiles:
        for b in (t - 1, t, t + 1, (M // t) * t - 1, (M // t) * t):
            if 0 <= b < M:
                rows.add(b)
    rng = np.random.default_rng(seed)
    rows.update(int(r) for r in rng.integers(0, M, size=count))
    return np.array(sorted(rows))


def oracle_fmaf_rows(A: np.ndarray, B: np.ndarray, rows: np.ndarray, N: int, K: int) -> np.ndarray:
    Asub = np.ascontiguousarray(A[rows])
    return oracle.gemm_fmaf_chain(Asub, B, len(rows), N, K)


def oracle_f64_rows(A: np.ndarray, B: np.ndarray, rows: np.ndarray, N: int, K: int) -> np.ndarray:
    Asub = np.ascontiguousarray(A[rows])
    return oracle.gemm_f64(Asub, B, len(rows), N, K)


def oracle_bf16_rows(A: np.ndarray, B: np.ndarray, rows: np.ndarray, N: int, K: int) -> np.ndarray:
    Asub = np.ascontiguousarray(A[rows])
    return oracle.gemm_bf16_f64(Asub, B, len(rows), N, K)


def bits(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)


def assert_bitwise_equal(got: np.ndarray, want: np.ndarray, what: str):
    gb, wb = bits(got), bits(want)
    if not np.array_equal(gb, wb):
        bad = np.argwhere(gb != wb)
        i, j = bad[0]
        raise AssertionError(f"{what}: {len(bad)} elements differ; first at ({i},{j}): "
                             f"got {got[i, j]!r} want {want[i, j]!r}")


def tma_pitch(n: int) -> int:
    """Smallest leading dimension >= n whose row pitch is a multiple of 16 bytes
    (what a TMA tensor map needs for float32 rows)."""
    return max(4, (n + 3) // 4 * 4)


def f32_operands(kind: str, M: int, N: int, K: int, seed: int, lda: int | None = None, ldb: int | None = None,
                 fill: str | None = None):
    """Seeded A (M x K) and B (K x N).  For the TMA fill the leading dimensions
    are raised to the nearest 16-byte row pitch (the same logical values; the
    extra columns are NaN padding)."""
    if fill == "tma":
        lda = tma_pitch(lda or K)
        ldb = tma_pitch(ldb or N)
    A = inputs.matrix_f32(kind, M, K, seed, inputs.TAG_A, ld=lda)
    B = inputs.matrix_f32(kind, K, N, seed, inputs.TAG_B, ld=ldb)
    return A, B


def bf16_pitch(n: int) -> int:
    """Smallest leading dimension >= n whose row pitch is a multiple of 16 bytes
    for bfloat16 rows."""
    return max(8, (n + 7) // 8 * 8)


def bf16_operands(kind: str, M: int, N: int, K: int, seed: int, sigma: float = 0.5,
                  lda: int | None = None, ldb: int | None = None):
    """Seeded bfloat16 A (M x K) and B (K x N) at 16-byte row pitches."""
    A = inputs.matrix_bf16(kind, M, K, seed, inputs.TAG_A, ld=bf16_pitch(lda or K), sigma=sigma)
    B = inputs.matrix_bf16(kind, K, N, seed, inputs.TAG_B, ld=bf16_pitch(ldb or N), sigma=sigma)
    return A, B
