"""The GEMM kernels' own bounded waits, made to expire without faulting,
trapping or hanging the GPU.

A test hook (include/pipelined_gemm_testing.h) makes the producers of one
kernel leave one ring position unfilled: no copy, no arrival, and for TMA no
expected-transaction count either, so no copy is ever in flight against a
barrier nobody armed.  That is the stranded block of "Day 74: Async copies and
pipelines", section "Pitfalls" (a missing commit leaves the waiters waiting).
With a 10 ms limit every wait on that position gives up; each call must
return, record GEMM_ERR_TIMEOUT with the kernel's family and a waiting role
(never the drain of copies or MMAs still in flight, which always land), and
leave the context able to compute the next GEMM exactly.

Every wait the hook reaches is bounded, each call ends in tens of
milliseconds, and the hook is reset after every case even when it fails.
"""
import numpy as np
import pytest

from gpu_util import assert_bitwise_equal, bf16_operands, f32_operands, run_bf16, run_f32

import oracle

pytestmark = pytest.mark.gpu

TIMEOUT = 6
FAMILY = {"f32_tma": 1, "bf16": 2, "f32_cpasync_mbar": 4, "f32_cpasync_ws": 5}
ROLE_DRAIN = 5
LIMIT_NS = 10_000_000  # 10 ms


@pytest.fixture
def hooks():
    import async_copy_pipelined_gb300 as pg
    assert pg.device_status()[0] == 0, "status word not clean before the case"
    yield pg
    pg.testing_set_hooks(0, -1)
    pg.device_status()  # leave the word clean for the next test


def _expect_timeout(pg, family: int, what: str):
    st, detail = pg.device_status()
    assert st == TIMEOUT, f"{what}: expected GEMM_ERR_TIMEOUT, got status {st} ({detail:#x})"
    assert detail & 0xFF == family, f"{what}: family {detail & 0xFF}, expected {family} ({detail:#x})"
    role = (detail >> 8) & 0xFF
    assert role in (1, 2, 3, 4), f"{what}: role {role} ({detail:#x})"
    assert role != ROLE_DRAIN, f"{what}: a drain wait expired ({detail:#x})"


F32_CASES = [("tma", 2, 128), ("tma", 4, 128), ("tma", 6, 128), ("tma", 3, 64), ("tma", 2, 32), ("tma", 6, 32),
             ("cpasync_mbar", 2, 128), ("cpasync_mbar", 4, 128), ("cpasync_mbar", 3, 64),
             ("cpasync_mbar", 2, 32), ("cpasync_mbar", 6, 32),
             ("cpasync_ws", 2, 128), ("cpasync_ws", 4, 128), ("cpasync_ws", 3, 64), ("cpasync_ws", 2, 32),
             ("cpasync_ws", 6, 32)]


@pytest.mark.parametrize("withhold", [0, 1, 7])
@pytest.mark.parametrize("fill,stages,tile", F32_CASES)
def test_f32_withheld_slice_times_out_then_exact(hooks, fill, stages, tile, withhold):
    pg = hooks
    import torch
    M, N, K = 2 * tile, 2 * tile, 8 * 16  # four CTAs, eight K slices
    A, B = f32_operands("uniform", M, N, K, seed=11)
    Ad = torch.from_numpy(A).cuda()[:, :K]
    Bd = torch.from_numpy(B).cuda()[:, :N]
    pg.testing_set_hooks(LIMIT_NS, withhold)
    pg.gemm_f32(Ad, Bd, fill=fill, stages=stages, block_tile=tile)
    _expect_timeout(pg, FAMILY["f32_" + fill], f"{fill} S{stages} T{tile} withhold {withhold}")
    pg.testing_set_hooks(0, -1)
    got, _ = run_f32(A, B, M, N, K, fill, stages, tile)
    assert_bitwise_equal(got, oracle.gemm_fmaf_chain(A, B, M, N, K), f"{fill} S{stages} T{tile} after timeout")


BF16_CASES = [("tma", 2, 128), ("tma", 4, 128), ("tma", 2, 256), ("tma", 3, 256), ("cpasync", 2, 128),
              ("cpasync", 4, 128), ("cpasync", 3, 256), ("sync", 1, 128), ("sync", 1, 256)]


@pytest.mark.parametrize("withhold", [0, 1, 4])
@pytest.mark.parametrize("fill,stages,block_m", BF16_CASES)
def test_bf16_withheld_stage_times_out_then_exact(hooks, fill, stages, block_m, withhold):
    """Every role of the persistent tensor-core kernel gives up in turn: the
    MMA issuer on the unfilled stage, the producers on a stage never
    released, the epilogue on an accumulator never completed.  The MMA issuer
    still waits for its own MMAs and for the epilogue before freeing tensor
    memory.  Four tiles, one per CTA, five K blocks each: the first, second
    and last position of the ring are withheld in turn."""
    pg = hooks
    import torch
    M, N, K = 2 * block_m, 512, 5 * 64
    A, B = bf16_operands("smallint", M, N, K, seed=12)
    Ad = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16).cuda()[:, :K]
    Bd = torch.from_numpy(B.view(np.int16)).view(torch.bfloat16).cuda()[:, :N]
    pg.testing_set_hooks(LIMIT_NS, withhold)
    pg.gemm_bf16(Ad, Bd, fill=fill, stages=stages, block_m=block_m)
    _expect_timeout(pg, FAMILY["bf16"], f"bf16 {fill} S{stages} T{block_m} withhold {withhold}")
    pg.testing_set_hooks(0, -1)
    got, _ = run_bf16(A, B, M, N, K, stages=stages, fill=fill, block_m=block_m)
    assert_bitwise_equal(got, oracle.gemm_bf16_f64(A, B, M, N, K).astype(np.float32),
                         f"bf16 {fill} S{stages} T{block_m} after timeout")


@pytest.mark.parametrize("fill,stages,block_m", [("tma", 4, 128), ("cpasync", 3, 256), ("sync", 1, 128)])
def test_bf16_withheld_stage_in_a_later_tile(hooks, fill, stages, block_m):
    """More tiles than SMs, so persistent CTAs walk several tiles: the
    unfilled position lies in a CTA's second tile, after its first tile's
    accumulator has gone through the epilogue."""
    pg = hooks
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M, N, K = block_m * 2 * ((sms + 1) // 2 + 1), 512, 2 * 64  # > sms tiles of two K blocks
    A, B = bf16_operands("smallint", M, N, K, seed=13)
    Ad = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16).cuda()[:, :K]
    Bd = torch.from_numpy(B.view(np.int16)).view(torch.bfloat16).cuda()[:, :N]
    pg.testing_set_hooks(LIMIT_NS, 3)  # second K block of the second tile
    pg.gemm_bf16(Ad, Bd, fill=fill, stages=stages, block_m=block_m)
    _expect_timeout(pg, FAMILY["bf16"], f"bf16 {fill} later tile")
    pg.testing_set_hooks(0, -1)
    got, _ = run_bf16(A, B, M, N, K, stages=stages, fill=fill, block_m=block_m)
    assert_bitwise_equal(got, oracle.gemm_bf16_f64(A, B, M, N, K).astype(np.float32), f"bf16 {fill} after")


def test_short_limit_alone_changes_nothing(hooks):
    """The short limit with no position withheld: normal calls still finish
    and still give the oracle's bits."""
    pg = hooks
    pg.testing_set_hooks(LIMIT_NS, -1)
    M, N, K = 300, 260, 200
    A, B = f32_operands("uniform", M, N, K, seed=14, fill="tma")
    for fill, stages, tile in (("tma", 4, 128), ("cpasync_mbar", 3, 64)):
        got, _ = run_f32(A, B, M, N, K, fill, stages, tile)
        assert_bitwise_equal(got, oracle.gemm_fmaf_chain(A, B, M, N, K), f"{fill} with a 10 ms limit")
