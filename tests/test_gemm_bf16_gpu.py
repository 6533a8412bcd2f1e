"""GPU parity of the BF16 tensor-core path against the oracle, through the C ABI.

The tensor core sums in its own order, so results are compared with the
exact-product float64 oracle within a tolerance: the acceptance bound
||C - C_ref||_F / ||C_ref||_F <= 2e-2, and the much tighter per-element bound
|C - C_ref| <= K * 2^-22 * sum_k |a_ik b_kj| that float32 accumulation of
exact products satisfies.  Small-integer inputs and the identity / all-ones
closed forms are exact in any order and are compared bit for bit.
"""
import numpy as np
import pytest

from async_copy_pipelined_gb300 import inputs
from gpu_util import bf16_operands, oracle_bf16_rows, run_bf16, sample_rows

import oracle

pytestmark = pytest.mark.gpu


def _abs_products(A, B, M, N, K):
    Aa = np.abs(inputs.bf16_bits_to_f32(A[:, :K])).astype(np.float64)
    Ba = np.abs(inputs.bf16_bits_to_f32(B[:, :N])).astype(np.float64)
    return Aa @ Ba


def _check(got, want, absprod, K, what):
    fro = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300)
    assert fro <= 2e-2, f"{what}: relative Frobenius error {fro}"
    bound = K * 2.0 ** -22 * absprod
    excess = np.abs(got - want) - bound
    assert np.all(excess <= 0), f"{what}: per-element bound exceeded by {excess.max()}"


SHAPES = [(1, 1, 1), (128, 256, 64), (128, 256, 128), (130, 300, 70), (64, 512, 200), (257, 513, 129),
          (300, 257, 1000), (1, 700, 64), (700, 1, 64)]


# (fill, stages, rows per CTA tile): every ring depth each tile holds.
BF16_CASES = [("tma", 2, 128), ("tma", 3, 128), ("tma", 4, 128), ("cpasync", 2, 128), ("cpasync", 3, 128),
              ("cpasync", 4, 128), ("sync", 1, 128),
              ("tma", 2, 256), ("tma", 3, 256), ("cpasync", 2, 256), ("cpasync", 3, 256), ("sync", 1, 256)]


@pytest.mark.parametrize("fill,stages,block_m", BF16_CASES)
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_small_ragged_normal(fill, stages, block_m, M, N, K):
    A, B = bf16_operands("normal", M, N, K, 60 + K)
    got, _ = run_bf16(A, B, M, N, K, stages=stages, fill=fill, block_m=block_m)
    want = oracle.gemm_bf16_f64(A, B, M, N, K)
    _check(got, want, _abs_products(A, B, M, N, K), K, f"bf16 {fill} S{stages} T{block_m} {M}x{N}x{K}")
    # Every fill and tile feeds the same MMA sequence per output element with
    # the same bytes: same bits.
    if (fill, stages, block_m) != ("tma", 4, 128):
        ref, _ = run_bf16(A, B, M, N, K, stages=4, fill="tma", block_m=128)
        np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32))


_WALK_CACHE = {}


def _walk_case(M, N, K):
    """Operands and oracle for a shape with more 128 x 256 tiles than SMs (so
    persistent CTAs walk several tiles), cached across fills."""
    key = (M, N, K)
    if key not in _WALK_CACHE:
        A, B = bf16_operands("normal", M, N, K, 70 + K)
        want = oracle.gemm_bf16_f64(A, B, M, N, K)
        ref, _ = run_bf16(A, B, M, N, K, stages=4, fill="tma", block_m=128)
        _WALK_CACHE[key] = (A, B, want, ref, _abs_products(A, B, M, N, K))
    return _WALK_CACHE[key]


@pytest.mark.parametrize("fill,stages,block_m", BF16_CASES)
@pytest.mark.parametrize("M,N,K", [(2048, 2560, 192), (2000, 2600, 200), (4096, 2560, 192), (4000, 2600, 200)])
def test_persistent_walk_interior_and_edge_tiles(fill, stages, block_m, M, N, K):
    """More tiles than the 152 persistent CTAs: 160 / 176 128-row tiles for
    the first two shapes, 160 / 176 256-row tiles for the last two.  The
    first shape of each pair has only interior tiles and whole K blocks (the
    thread-issued fills' per-tile address path throughout); the second mixes
    interior and edge tiles and ends every tile with an 8-deep K tail
    (guarded path for edge tiles and for the last K block)."""
    A, B, want, ref, absprod = _walk_case(M, N, K)
    got, _ = run_bf16(A, B, M, N, K, stages=stages, fill=fill, block_m=block_m)
    _check(got, want, absprod, K, f"bf16 {fill} S{stages} T{block_m} {M}x{N}x{K}")
    np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("fill,stages,block_m", [("tma", 4, 128), ("cpasync", 3, 128), ("sync", 1, 128),
                                                 ("tma", 3, 256), ("cpasync", 2, 256), ("sync", 1, 256)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 300, 500), (513, 257, 1000)])
def test_smallint_exact(fill, stages, block_m, M, N, K):
    A, B = bf16_operands("smallint", M, N, K, 8)
    got, _ = run_bf16(A, B, M, N, K, stages=stages, fill=fill, block_m=block_m)
    Ai = inputs.bf16_bits_to_f32(A[:, :K]).astype(np.int64)
    Bi = inputs.bf16_bits_to_f32(B[:, :N]).astype(np.int64)
    np.testing.assert_array_equal(got, (Ai @ Bi).astype(np.float32))


def test_closed_forms():
    M = N = K = 256
    B = inputs.matrix_bf16("normal", K, N, 3, inputs.TAG_B, sigma=0.5)
    ident = inputs.matrix_bf16("identity", M, K, 0, 0)
    got, _ = run_bf16(ident, B, M, N, K)
    np.testing.assert_array_equal(got, inputs.bf16_bits_to_f32(B))
    A = inputs.matrix_bf16("normal", M, K, 3, inputs.TAG_A, sigma=0.5)
    got, _ = run_bf16(A, inputs.matrix_bf16("identity", K, N, 0, 0), M, N, K)
    np.testing.assert_array_equal(got, inputs.bf16_bits_to_f32(A))
    ones_a = inputs.matrix_bf16("ones", M, K, 0, 0)
    ones_b = inputs.matrix_bf16("ones", K, N, 0, 0)
    got, _ = run_bf16(ones_a, ones_b, M, N, K)
    assert np.all(got == np.float32(K))


@pytest.mark.parametrize("block_m", [128, 256])
@pytest.mark.parametrize("ldc_pad", [3, 4, 36])
def test_padded_and_ldc_canary(block_m, ldc_pad):
    """Padded operands, and C rows longer than N: with ldc = N + 3 rows are
    not 16-byte aligned and the epilogue stores element by element; with
    N + 4 and N + 36 the TMA stores must clip at column N.  The padding
    columns must keep their sentinel."""
    M, N, K = 300, 300, 96
    A, B = bf16_operands("normal", M, N, K, 5, lda=K + 8, ldb=N + 16)
    got, full = run_bf16(A, B, M, N, K, ldc=N + ldc_pad, sentinel=-5.0, block_m=block_m)
    want = oracle.gemm_bf16_f64(A, B, M, N, K)
    _check(got, want, _abs_products(A, B, M, N, K), K, f"padded T{block_m} ldc N+{ldc_pad}")
    assert np.all(full[:, N:] == -5.0)


def test_empty_and_k_zero():
    import torch
    import async_copy_pipelined_gb300 as pg
    C = torch.full((3, 9), 4.0, device="cuda")
    pg.gemm_bf16(torch.empty((3, 0), dtype=torch.bfloat16, device="cuda"),
                 torch.empty((0, 9), dtype=torch.bfloat16, device="cuda"), C)
    assert torch.count_nonzero(C).item() == 0
    C = pg.gemm_bf16(torch.empty((0, 16), dtype=torch.bfloat16, device="cuda"),
                     torch.ones((16, 8), dtype=torch.bfloat16, device="cuda"))
    assert C.shape == (0, 8)
    assert pg.device_status()[0] == 0


def test_workload_8192_sampled():
    """The bf16 workload at full size in the bench's launch configuration,
    checked on sampled rows (every column) against the exact-product oracle."""
    import torch
    import async_copy_pipelined_gb300 as pg
    w = inputs.WORKLOADS["bf16_8192"]
    M, N, K = w["M"], w["N"], w["K"]
    A, B = inputs.workload_operands("bf16_8192")
    Ad = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16).cuda()
    Bd = torch.from_numpy(B.view(np.int16)).view(torch.bfloat16).cuda()
    C = pg.gemm_bf16(Ad, Bd)
    assert pg.device_status()[0] == 0
    rows = sample_rows(M, 12, seed=4, tiles=(128,))
    got = C.cpu().numpy()[rows]
    want = oracle_bf16_rows(A, B, rows, N, K)
    _check(got, want, _abs_products(np.ascontiguousarray(A[rows]), B, len(rows), N, K), K, "8192^3 sampled")
    # Repeat: the persistent schedule must give the same bits every run, and
    # the cp.async and register-path fills the same bits as the TMA fill.
    C2 = pg.gemm_bf16(Ad, Bd)
    assert torch.equal(C.view(torch.int32), C2.view(torch.int32))
    for fill, stages, block_m in (("tma", 4, 128), ("tma", 2, 256), ("cpasync", 4, 128), ("cpasync", 3, 256),
                                  ("cpasync", 2, 128), ("sync", 1, 128), ("sync", 1, 256)):
        C3 = pg.gemm_bf16(Ad, Bd, fill=fill, stages=stages, block_m=block_m)
        assert torch.equal(C.view(torch.int32), C3.view(torch.int32)), (fill, stages, block_m)
    assert pg.device_status()[0] == 0


def test_workload_8192_normal_whole_output():
    """The bf16 workload at full size (normal(0, 0.5) inputs, the bench's
    launch configuration) over the whole output: every element within the
    float32-accumulation bound of the exact-product oracle, and the relative
    Frobenius error within the acceptance bound."""
    import torch
    import async_copy_pipelined_gb300 as pg
    w = inputs.WORKLOADS["bf16_8192"]
    M, N, K = w["M"], w["N"], w["K"]
    A, B = inputs.workload_operands("bf16_8192")
    Ad = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16).cuda()
    Bd = torch.from_numpy(B.view(np.int16)).view(torch.bfloat16).cuda()
    got = pg.gemm_bf16(Ad, Bd)
    assert pg.device_status()[0] == 0
    got = got.cpu().numpy()
    del Ad, Bd
    want = oracle.gemm_bf16_f64(A, B, M, N, K)
    _check(got, want, _abs_products(A, B, M, N, K), K, "8192^3 normal, whole output")


def test_workload_8192_smallint_exact_whole_output():
    """Entries in {-2..2} at 8192^3: exact in bfloat16, and every partial sum
    is an integer of magnitude at most 4K < 2^24, so the FP32 accumulator is
    exact whatever order the tensor cores add in.  The whole output must
    equal the exact product, for every fill and both tiles."""
    M = N = K = 8192
    A, B = bf16_operands("smallint", M, N, K, 104)
    want = oracle.gemm_bf16_f64(A, B, M, N, K).astype(np.float32)
    for fill, stages, block_m in (("tma", 0, 0), ("tma", 4, 128), ("cpasync", 4, 128), ("cpasync", 3, 256),
                                  ("sync", 1, 256)):
        got, _ = run_bf16(A, B, M, N, K, stages=stages, fill=fill, block_m=block_m)
        np.testing.assert_array_equal(got, want, err_msg=f"8192^3 small-int {fill}/S{stages}/T{block_m}")


@pytest.mark.parametrize("fill,stages,block_m", [("tma", 4, 128), ("tma", 2, 128), ("cpasync", 3, 128),
                                                 ("sync", 1, 128), ("tma", 3, 256), ("cpasync", 2, 256),
                                                 ("sync", 1, 256)])
def test_randomized_shapes(fill, stages, block_m):
    """Random ragged sizes and padded leading dimensions (seeded); N mod 4
    decides whether C is written by TMA stores or by plain stores."""
    rng = np.random.default_rng(1234 + stages)
    for _ in range(8):
        M, N, K = (int(rng.integers(1, 400)), int(rng.integers(1, 600)), int(rng.integers(1, 300)))
        A, B = bf16_operands("normal", M, N, K, M + N + K, lda=K + int(rng.integers(0, 17)),
                             ldb=N + int(rng.integers(0, 17)))
        got, _ = run_bf16(A, B, M, N, K, stages=stages, fill=fill, block_m=block_m)
        want = oracle.gemm_bf16_f64(A, B, M, N, K)
        _check(got, want, _abs_products(A, B, M, N, K), K, f"bf16 {fill} S{stages} T{block_m} {M}x{N}x{K}")


@pytest.mark.parametrize("fill", ["tma", "cpasync"])
def test_host_tensors_chunked_match_device_path(fill):
    """BF16 host tensors: B first, then row chunks of A in, GEMM, rows of C
    out on three streams; the same bits as one device call, and within the
    float32-accumulation bound of the oracle."""
    import torch
    import async_copy_pipelined_gb300 as pg
    M, N, K = 2000, 4096, 136
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    chunks = pg.host_row_chunks(M, N, sms)
    assert len(chunks) > 1 and chunks[-1][1] == M
    A, B = bf16_operands("normal", M, N, K, 91)
    Ah = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16).pin_memory()[:, :K]
    Bh = torch.from_numpy(B.view(np.int16)).view(torch.bfloat16).pin_memory()[:, :N]
    Ch = pg.gemm_bf16(Ah, Bh, fill=fill)
    assert not Ch.is_cuda
    got, _ = run_bf16(A, B, M, N, K, fill=fill)
    np.testing.assert_array_equal(Ch.numpy().view(np.uint32), got.view(np.uint32))
    rows = sample_rows(M, 24, 92)
    want = oracle_bf16_rows(A, B, rows, N, K)
    _check(Ch.numpy()[rows], want, _abs_products(A[rows], B, len(rows), N, K), K, f"bf16 host path {fill}")
