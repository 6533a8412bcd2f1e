"""The FP32 TMA fill's split of the last round of 128 x 128 tiles between
CTAs (gemm_f32_ws: the one-tile kernel for the whole rounds, then a
persistent kernel for the split region), through the C ABI.

A tile split between two CTAs is computed in K order, the second CTA
continuing from the first one's FP32 accumulators, so every element is
still one fused multiply-add chain over k ascending from +0: the output
must equal the oracle's FMA chain bit for bit, with the split and without
it, whatever the number of slices each CTA gets.
"""
import ctypes

import numpy as np
import pytest

from gpu_util import assert_bitwise_equal, f32_operands, to_device

import oracle

pytestmark = pytest.mark.gpu

# (M, N, K): tile counts 208 (k = 5), 320 (k = 3), 336 (ragged M, N and a
# ragged last K slice), 153 (one tile over a round, k = 2), 1200 (k = 64),
# and 304 / 64 tiles (whole rounds only, nothing to split).
SHAPES = [(1600, 2048, 80), (2048, 2560, 48), (1999, 2571, 133), (153 * 128, 128, 17), (3840, 5120, 1024),
          (152 * 128, 256, 40), (1024, 1024, 300)]


def _run(A, B, M, N, K, stages, workspace="auto"):
    import torch
    import async_copy_pipelined_gb300 as pg
    C = pg.gemm_f32(to_device(A, K), to_device(B, N), fill="tma", stages=stages, block_tile=128,
                    workspace=workspace)
    st, detail = pg.device_status()
    assert st == 0, f"device status {st} ({detail:#x})"
    torch.cuda.synchronize()
    return C.cpu().numpy()


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_split_and_unsplit_equal_the_fma_chain(M, N, K):
    import async_copy_pipelined_gb300 as pg
    A, B = f32_operands("uniform", M, N, K, seed=31, fill="tma")
    want = oracle.gemm_fmaf_chain(A, B, M, N, K)
    plan = pg.plan_f32(M, N, K, lda=A.shape[1], ldb=B.shape[1], fill="tma", stages=4, block_tile=128)
    tiles = plan["grid_x"] * plan["grid_y"]
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert (plan["persistent_ctas"] > 0) == (tiles > sms and tiles % sms != 0 and plan["k_slices"] >= 2)
    for stages in (2, 4, 6):
        assert_bitwise_equal(_run(A, B, M, N, K, stages), want, f"{M}x{N}x{K} S{stages} split")
    assert_bitwise_equal(_run(A, B, M, N, K, 3, workspace=None), want, f"{M}x{N}x{K} unsplit")


def test_workspace_is_checked():
    """An explicit workspace: too small is refused, misaligned is refused,
    and one exactly as large as the plan asks for is used as given."""
    import torch
    import async_copy_pipelined_gb300 as pg
    M, N, K = 1600, 2048, 80
    A, B = f32_operands("uniform", M, N, K, seed=32, fill="tma")
    want = oracle.gemm_fmaf_chain(A, B, M, N, K)
    Ad, Bd = to_device(A, K), to_device(B, N)
    need = pg.plan_f32(M, N, K, lda=A.shape[1], ldb=B.shape[1], fill="tma", block_tile=128)["workspace_bytes"]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert need == sms * (128 * 128 * 4 + 8)
    C = torch.empty((M, N), device="cuda")
    lib = pg.lib()
    h = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ws = torch.zeros(need + 64, dtype=torch.uint8, device="cuda")
    args = (M, N, K, Ad.data_ptr(), Ad.stride(0), Bd.data_ptr(), Bd.stride(0), C.data_ptr(), N, 2, 4, 128)
    assert lib.gemm_f32_ws(*args, ws.data_ptr(), need - 1, h) == 1
    assert lib.gemm_f32_ws(*args, ws.data_ptr() + 4, need, h) == 2
    # garbage in the workspace does not matter: it holds nothing between calls
    ws.fill_(0xAB)
    assert lib.gemm_f32_ws(*args, ws.data_ptr(), need, h) == 0
    assert pg.device_status()[0] == 0
    assert_bitwise_equal(C.cpu().numpy(), want, "explicit workspace")
    # the same workspace again (flags from the previous call must not count)
    C.fill_(7.0)
    assert lib.gemm_f32_ws(*args, ws.data_ptr(), need, h) == 0
    assert pg.device_status()[0] == 0
    assert_bitwise_equal(C.cpu().numpy(), want, "workspace reused")


@pytest.fixture
def hooks():
    import async_copy_pipelined_gb300 as pg
    assert pg.device_status()[0] == 0
    yield pg
    pg.testing_set_hooks(0, -1)
    pg.lib().gemm_testing_withhold_handover(0)
    pg.device_status()


def test_handover_wait_times_out_then_exact(hooks):
    """Heads never raise their ready flag: every CTA waiting for one gives up
    after the limit and records the hand-over role (6); the context then
    computes the next GEMM exactly."""
    pg = hooks
    M, N, K = 1600, 2048, 80
    A, B = f32_operands("uniform", M, N, K, seed=33, fill="tma")
    pg.testing_set_hooks(10_000_000, -1)
    pg.lib().gemm_testing_withhold_handover(1)
    import torch
    pg.gemm_f32(to_device(A, K), to_device(B, N), fill="tma", stages=4, block_tile=128)
    st, detail = pg.device_status()
    assert st == 6 and detail & 0xFF == 1 and (detail >> 8) & 0xFF == 6, f"{st} {detail:#x}"
    pg.lib().gemm_testing_withhold_handover(0)
    pg.testing_set_hooks(0, -1)
    assert_bitwise_equal(_run(A, B, M, N, K, 4), oracle.gemm_fmaf_chain(A, B, M, N, K), "after hand-over timeout")
    torch.cuda.synchronize()


@pytest.mark.parametrize("withhold", [0, 1, 2])
def test_withheld_slice_in_a_split_schedule_times_out(hooks, withhold):
    """A ring position left unfilled in a split schedule (every CTA's own
    position `withhold`, in the whole-round kernel and in the split-region
    kernel, each CTA of which has at least three): the waits on it and on the
    hand-overs that can no longer come all end, and the next call is exact."""
    pg = hooks
    M, N, K = 2048, 2560, 48
    A, B = f32_operands("uniform", M, N, K, seed=34, fill="tma")
    pg.testing_set_hooks(10_000_000, withhold)
    pg.gemm_f32(to_device(A, K), to_device(B, N), fill="tma", stages=2, block_tile=128)
    st, detail = pg.device_status()
    assert st == 6 and detail & 0xFF == 1 and (detail >> 8) & 0xFF != 5, f"{st} {detail:#x}"
    pg.testing_set_hooks(0, -1)
    assert_bitwise_equal(_run(A, B, M, N, K, 2), oracle.gemm_fmaf_chain(A, B, M, N, K), "after timeout")
