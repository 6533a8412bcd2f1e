"""GPU parity of the FP32 kernel family against the oracle, through the C ABI.

The bar: every FP32 result equals the oracle's
float32 FMA chain bit for bit (hence all fills, stage counts and tiles are
bit-identical to each other, the pages' memcmp invariant), and lies within
max|C - C_ref| <= 1e-5 * K of the float64 definition.
"""
import zlib

import numpy as np
import pytest

from async_copy_pipelined_gb300 import inputs
from gpu_util import F32_VARIANTS, assert_bitwise_equal, f32_operands, run_f32, tma_pitch

import oracle

pytestmark = pytest.mark.gpu

SMALL_SHAPES = [
    (1, 1, 1), (1, 5, 3), (7, 1, 17), (16, 16, 16), (17, 33, 15), (64, 64, 16), (65, 63, 17),
    (128, 128, 32), (129, 130, 31), (130, 257, 100), (200, 150, 1000), (33, 300, 48),
]


def _check_against_oracle(A, B, M, N, K, got, what):
    want32 = oracle.gemm_fmaf_chain(A, B, M, N, K)
    assert_bitwise_equal(got, want32, what + " vs FMA-chain oracle")
    want64 = oracle.gemm_f64(A, B, M, N, K)
    err = np.max(np.abs(got.astype(np.float64) - want64)) if got.size else 0.0
    assert err <= 1e-5 * max(K, 1), f"{what}: max abs err {err} > 1e-5*K"


@pytest.mark.parametrize("fill,stages,tile", F32_VARIANTS)
@pytest.mark.parametrize("M,N,K", SMALL_SHAPES)
def test_small_ragged_uniform(fill, stages, tile, M, N, K):
    A, B = f32_operands("uniform", M, N, K, seed=100 + M + N + K, fill=fill)
    got, _ = run_f32(A, B, M, N, K, fill, stages, tile)
    _check_against_oracle(A, B, M, N, K, got, f"{fill}/S{stages}/T{tile} {M}x{N}x{K}")


@pytest.mark.parametrize("fill,stages,tile", F32_VARIANTS)
def test_padded_leading_dims_and_ldc_canary(fill, stages, tile):
    """lda > K and ldb > N with NaN padding (a read of padding poisons C) and
    ldc > N with a sentinel that must survive."""
    M, N, K = 150, 130, 77
    lda, ldb, ldc = (K + 3 if fill != "tma" else K + 7), N + 6, N + 5
    A, B = f32_operands("normal", M, N, K, seed=7, lda=lda, ldb=ldb, fill=fill)
    got, full = run_f32(A, B, M, N, K, fill, stages, tile, ldc=ldc, sentinel=-777.0)
    _check_against_oracle(A, B, M, N, K, got, f"{fill}/S{stages}/T{tile} padded")
    assert np.all(full[:, N:] == -777.0), "columns beyond N were written"


@pytest.mark.parametrize("fill,stages,tile", F32_VARIANTS)
def test_smallint_exact(fill, stages, tile):
    """Small integers: the product is exact in any order and must equal
    numpy's int64 matmul."""
    M, N, K = 97, 131, 300
    A, B = f32_operands("smallint", M, N, K, seed=5, fill=fill)
    got, _ = run_f32(A, B, M, N, K, fill, stages, tile)
    want = (A[:, :K].astype(np.int64) @ B[:, :N].astype(np.int64)).astype(np.float32)
    np.testing.assert_array_equal(got, want)


# ----------------------------------------------------- workload 1: 256^3

def test_workload_256_all_fills_and_closed_forms():
    w = inputs.WORKLOADS["f32_256"]
    M, N, K = w["M"], w["N"], w["K"]
    A, B = inputs.workload_operands("f32_256")
    want32 = oracle.gemm_fmaf_chain(A, B, M, N, K)
    want64 = oracle.gemm_f64(A, B, M, N, K)
    for fill, stages, tile in F32_VARIANTS:
        got, _ = run_f32(A, B, M, N, K, fill, stages, tile)
        assert_bitwise_equal(got, want32, f"256^3 {fill}/S{stages}/T{tile}")
        assert np.max(np.abs(got - want64)) <= 1e-5 * K
    ident = inputs.matrix_f32("identity", M, K, 0, 0)
    ones_a = inputs.matrix_f32("ones", M, K, 0, 0)
    ones_b = inputs.matrix_f32("ones", K, N, 0, 0)
    for fill, stages, tile in [("sync", 1, 64), ("cpasync", 2, 64), ("tma", 2, 64), ("tma", 4, 128)]:
        got, _ = run_f32(ident, B, M, N, K, fill, stages, tile)
        np.testing.assert_array_equal(got, B, err_msg=f"I*B != B ({fill})")
        got, _ = run_f32(A, ident, M, N, K, fill, stages, tile)
        np.testing.assert_array_equal(got, A, err_msg=f"A*I != A ({fill})")
        got, _ = run_f32(ones_a, ones_b, M, N, K, fill, stages, tile)
        assert np.all(got == np.float32(K)), f"ones*ones != K ({fill})"
        got, _ = run_f32(A, ones_b, M, N, K, fill, stages, tile)
        # Row sums: every column equals the sequential float32 sum of the row.
        rowsum = oracle.gemm_fmaf_chain(A, ones_b[:, :1].copy(), M, 1, K)
        assert np.all(got == rowsum), f"row sums differ ({fill})"


# ----------------------------------------------------- workload 2: 1024^3

def test_workload_1024_fills_bit_identical():
    w = inputs.WORKLOADS["f32_1024"]
    M, N, K = w["M"], w["N"], w["K"]
    A, B = inputs.workload_operands("f32_1024")
    want32 = oracle.gemm_fmaf_chain(A, B, M, N, K)
    want64 = oracle.gemm_f64(A, B, M, N, K)
    outs = {}
    for fill, stages, tile in [("sync", 1, 64), ("cpasync", 2, 64), ("tma", 2, 64), ("sync", 1, 128),
                               ("cpasync", 4, 128), ("tma", 4, 128), ("cpasync_mbar", 2, 64),
                               ("cpasync_mbar", 4, 128), ("cpasync_ws", 2, 64), ("cpasync_ws", 4, 128)]:
        got, _ = run_f32(A, B, M, N, K, fill, stages, tile)
        outs[(fill, stages, tile)] = got
        assert_bitwise_equal(got, want32, f"1024^3 {fill}/S{stages}/T{tile}")
    err = np.max(np.abs(outs[("sync", 1, 64)] - want64))
    assert err <= 1e-5 * K
    base = outs[("sync", 1, 64)].view(np.uint32)
    for key, v in outs.items():
        assert np.array_equal(v.view(np.uint32), base), f"{key} differs from the sync fill"


# ----------------------------------------------------- workload 3: 4096^3

def test_workload_4096_stage_sweep_whole_output():
    """Full-size config in the bench's launch configuration: every fill and
    stage count bitwise equal to each other, and to the oracle's FMA chain,
    over the whole output."""
    import torch
    import async_copy_pipelined_gb300 as pg
    w = inputs.WORKLOADS["f32_4096"]
    M, N, K = w["M"], w["N"], w["K"]
    A, B = inputs.workload_operands("f32_4096")
    Ad = torch.from_numpy(A).cuda()
    Bd = torch.from_numpy(B).cuda()
    ref = pg.gemm_f32(Ad, Bd, fill="sync", block_tile=128)
    for fill, stages in [("cpasync", 2), ("cpasync", 3), ("cpasync", 4), ("cpasync", 6),
                         ("tma", 2), ("tma", 3), ("tma", 4), ("tma", 6), ("cpasync_mbar", 2), ("cpasync_mbar", 4),
                         ("cpasync_mbar", 6), ("cpasync_ws", 2), ("cpasync_ws", 4), ("cpasync_ws", 6)]:
        out = pg.gemm_f32(Ad, Bd, fill=fill, stages=stages, block_tile=128)
        assert torch.equal(out.view(torch.int32), ref.view(torch.int32)), f"{fill}/S{stages} != sync"
    out64 = pg.gemm_f32(Ad, Bd, fill="tma", stages=4, block_tile=64)
    assert torch.equal(out64.view(torch.int32), ref.view(torch.int32)), "64-tile TMA != sync"
    assert pg.device_status()[0] == 0
    got = ref.cpu().numpy()
    assert_bitwise_equal(got, oracle.gemm_fmaf_chain(A, B, M, N, K), "4096^3 whole output")
    assert np.max(np.abs(got - oracle.gemm_f64(A, B, M, N, K))) <= 1e-5 * K


# ----------------------------------------------------- workload 4: ragged

def test_workload_ragged_lda_k_plus_3():
    """M=3000 N=5000 K=1000, lda=1003 (rows not 16-byte aligned): sync and
    cp.async read A with 4-byte copies; TMA cannot describe that pitch and
    must refuse it; the same logical A repacked at lda=1004 runs through TMA
    and must give the same bits."""
    import torch
    import async_copy_pipelined_gb300 as pg
    w = inputs.WORKLOADS["f32_ragged"]
    M, N, K = w["M"], w["N"], w["K"]
    A, B = inputs.workload_operands("f32_ragged")
    assert A.shape == (M, 1003)
    Ad = torch.from_numpy(A).cuda()[:, :K]
    Bd = torch.from_numpy(B).cuda()
    plan = pg.plan_f32(M, N, K, lda=1003, fill="cpasync")
    assert plan["a_copy_bytes"] == 4 and plan["b_copy_bytes"] == 16
    outs = {}
    for fill, stages, tile in [("sync", 1, 64), ("sync", 1, 128), ("cpasync", 2, 64), ("cpasync", 3, 128),
                               ("cpasync", 6, 128), ("cpasync_mbar", 3, 128), ("cpasync_mbar", 2, 64)]:
        outs[(fill, stages, tile)] = pg.gemm_f32(Ad, Bd, fill=fill, stages=stages, block_tile=tile)
    with pytest.raises(pg.GemmError) as e:
        pg.gemm_f32(Ad, Bd, fill="tma", stages=4)
    assert e.value.status == 2  # GEMM_ERR_MISALIGNED
    A4 = inputs.workload_operands("f32_ragged", lda=1004)[0]
    Ad4 = torch.from_numpy(A4).cuda()[:, :K]
    for stages, tile in [(2, 64), (4, 128), (6, 128)]:
        outs[("tma", stages, tile)] = pg.gemm_f32(Ad4, Bd, fill="tma", stages=stages, block_tile=tile)
    assert pg.device_status()[0] == 0
    ref = outs[("sync", 1, 64)]
    for key, v in outs.items():
        assert torch.equal(v.view(torch.int32), ref.view(torch.int32)), f"{key} differs from sync"
    got = ref.cpu().numpy()
    assert_bitwise_equal(got, oracle.gemm_fmaf_chain(A, B, M, N, K), "ragged whole output")
    assert np.max(np.abs(got - oracle.gemm_f64(A, B, M, N, K))) <= 1e-5 * K


# ----------------------------------------------------- small integers at every workload's shape

@pytest.mark.parametrize("name", ["f32_256", "f32_1024", "f32_4096", "f32_ragged"])
def test_workload_shapes_smallint_exact(name):
    """Entries in {-2..2} at the workload's own sizes and leading dimension.
    Every partial sum is an integer of magnitude at most 4K < 2^24, so the
    product is exact in any order: every fill must equal the exact product
    over the whole output (the TMA fill reads the same values at the next
    16-byte row pitch when lda is not one)."""
    w = inputs.WORKLOADS[name]
    M, N, K, lda = w["M"], w["N"], w["K"], w["lda"]
    seed = 100 + w["seed"]
    A = inputs.matrix_f32("smallint", M, K, seed, inputs.TAG_A, ld=lda)
    B = inputs.matrix_f32("smallint", K, N, seed, inputs.TAG_B)
    A4 = A if lda % 4 == 0 else inputs.matrix_f32("smallint", M, K, seed, inputs.TAG_A, ld=tma_pitch(lda))
    want = oracle.gemm_f64(A, B, M, N, K).astype(np.float32)
    for fill, stages in (("sync", 1), ("cpasync", 3), ("cpasync_mbar", 4), ("tma", 4)):
        got, _ = run_f32(A4 if fill == "tma" else A, B, M, N, K, fill, stages, 0)
        np.testing.assert_array_equal(got, want, err_msg=f"{name} {fill}/S{stages}")


# ----------------------------------------------------- tall K, one warp

def test_workload_tallk_one_warp_all_fills():
    """M = N = 32, K = 65536 on the one-warp 32x32 tile: every fill and stage
    count equals the oracle's FMA chain bit for bit (4096 slices each)."""
    w = inputs.WORKLOADS["f32_tallk"]
    M, N, K = w["M"], w["N"], w["K"]
    A, B = inputs.workload_operands("f32_tallk")
    want32 = oracle.gemm_fmaf_chain(A, B, M, N, K)
    want64 = oracle.gemm_f64(A, B, M, N, K)
    for fill, stages in [("sync", 1), ("cpasync", 2), ("cpasync", 4), ("cpasync", 6), ("tma", 2), ("tma", 4),
                         ("tma", 6), ("cpasync_mbar", 2), ("cpasync_mbar", 4), ("cpasync_mbar", 6)]:
        got, _ = run_f32(A, B, M, N, K, fill, stages, 32)
        assert_bitwise_equal(got, want32, f"tall-K {fill}/S{stages}")
    assert np.max(np.abs(got - want64)) <= 1e-5 * K


# ----------------------------------------------------- edge cases

@pytest.mark.parametrize("fill", ["sync", "cpasync", "tma", "cpasync_mbar"])
def test_empty_sizes(fill):
    import torch
    import async_copy_pipelined_gb300 as pg
    # M == 0 and N == 0: no-op.
    C = pg.gemm_f32(torch.empty((0, 8), device="cuda"), torch.ones((8, 4), device="cuda"), fill=fill)
    assert C.shape == (0, 4)
    C = pg.gemm_f32(torch.ones((4, 8), device="cuda"), torch.empty((8, 0), device="cuda"), fill=fill)
    assert C.shape == (4, 0)
    # K == 0: an empty sum, C is all zeros (overwriting whatever was there).
    C = torch.full((5, 7), 3.0, device="cuda")
    pg.gemm_f32(torch.empty((5, 0), device="cuda"), torch.empty((0, 7), device="cuda"), C, fill=fill)
    assert torch.count_nonzero(C).item() == 0
    assert pg.device_status()[0] == 0


def test_page4_pattern_all_fills():
    """The lesson program's own inputs at its first size, N = 512."""
    n = 512
    a = inputs.matrix_f32("page4a", n, n, 0, 0)
    b = inputs.matrix_f32("page4b", n, n, 0, 0)
    want = oracle.gemm_fmaf_chain(a, b, n, n, n)
    want64 = oracle.gemm_f64(a, b, n, n, n)
    for fill, stages, tile in [("sync", 1, 64), ("cpasync", 2, 64), ("tma", 2, 64), ("tma", 4, 128),
                               ("cpasync_mbar", 2, 64)]:
        got, _ = run_f32(a, b, n, n, n, fill, stages, tile)
        assert_bitwise_equal(got, want, f"page-4 pattern {fill}")
        # The program's own relative check (rel 1e-4, scale 1 at zero) holds too.
        scale = np.where(want64 == 0, 1.0, np.abs(want64))
        assert np.all(np.abs(got - want64) <= 1e-4 * scale)


def test_non_default_stream():
    import torch
    import async_copy_pipelined_gb300 as pg
    M, N, K = 300, 200, 100
    A, B = f32_operands("uniform", M, N, K, seed=44)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        Ad = torch.from_numpy(A).cuda()
        Bd = torch.from_numpy(B).cuda()
        C = pg.gemm_f32(Ad, Bd, fill="tma", stages=3, stream=s)
    s.synchronize()
    assert_bitwise_equal(C.cpu().numpy(), oracle.gemm_fmaf_chain(A, B, M, N, K), "side stream")


@pytest.mark.parametrize("fill", ["sync", "tma"])
def test_host_tensors_chunked_match_device_path(fill):
    """A host call (the native executor, one K block at this K) split into
    several row chunks, the last one ragged, gives the same bits as one
    device call."""
    import torch
    import async_copy_pipelined_gb300 as pg
    M, N, K = 3300, 4096, 256
    A, B = f32_operands("uniform", M, N, K, seed=10, fill="tma")
    Ah = torch.from_numpy(A).pin_memory()[:, :K]
    Bh = torch.from_numpy(B).pin_memory()[:, :N]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    kb, rb = pg.host_schedule_f32(M, N, K, sms)
    assert kb == [0, K] and len(rb) > 3 and (rb[-1] - rb[-2]) % 128
    Ch = pg.gemm_f32(Ah, Bh, fill=fill)
    Cd = pg.gemm_f32(torch.from_numpy(A).cuda()[:, :K], torch.from_numpy(B).cuda()[:, :N], fill=fill)
    assert torch.equal(Ch.view(torch.int32), Cd.cpu().view(torch.int32))
    assert_bitwise_equal(Ch.numpy(), oracle.gemm_fmaf_chain(A, B, M, N, K), "chunked host path")


def test_host_tensors_end_to_end():
    import torch
    import async_copy_pipelined_gb300 as pg
    M, N, K = 129, 65, 40
    A, B = f32_operands("uniform", M, N, K, seed=9)
    C = pg.gemm_f32(torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory(), fill="cpasync")
    assert not C.is_cuda
    assert_bitwise_equal(C.numpy(), oracle.gemm_fmaf_chain(A, B, M, N, K), "host round trip")


# ----------------------------------------------------- randomized shapes

def _random_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        M = int(rng.integers(1, 300))
        N = int(rng.integers(1, 300))
        K = int(rng.integers(1, 200))
        pad_a = int(rng.integers(0, 9))
        pad_b = int(rng.integers(0, 9))
        cases.append((M, N, K, pad_a, pad_b))
    return cases


@pytest.mark.parametrize("fill,stages,tile", [("sync", 1, 64), ("sync", 1, 128), ("cpasync", 3, 64),
                                              ("cpasync", 5, 128), ("cpasync_mbar", 2, 32),
                                              ("cpasync_mbar", 4, 128), ("tma", 2, 32), ("tma", 3, 64),
                                              ("tma", 6, 128)])
def test_randomized_shapes(fill, stages, tile):
    """Random ragged sizes and leading-dimension padding, every result bitwise
    equal to the oracle's FMA chain (seeded, so failures reproduce)."""
    for M, N, K, pad_a, pad_b in _random_cases(12, seed=zlib.crc32(f"{fill}/{stages}/{tile}".encode())):
        A, B = f32_operands("normal", M, N, K, seed=M * 7 + N * 3 + K, lda=K + pad_a, ldb=N + pad_b, fill=fill)
        got, _ = run_f32(A, B, M, N, K, fill, stages, tile)
        assert_bitwise_equal(got, oracle.gemm_fmaf_chain(A, B, M, N, K),
                             f"{fill}/S{stages}/T{tile} {M}x{N}x{K} pads {pad_a},{pad_b}")
