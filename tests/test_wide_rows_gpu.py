"""The TMA fill's wide-row kernel (128 x 256 tiles, 8 x 16 micro-tile, copies
issued by a consumer thread): the top rows of a call on the 128 tile, when
the planner gives it any (gemm_plan.wide_rows), the 128 x 128 path below.

Every element is still one FMA chain over k ascending, so each call must
equal the oracle's FMA chain bit for bit: with the wide kernel taking all
rows, some rows (the split 128 x 128 path computing the rest), or none (the
testing knob off), with ragged M, N and K edges, with accumulation from C,
and after a withheld ring position made its waits run out.
"""
import numpy as np
import pytest

from gpu_util import assert_bitwise_equal, f32_operands, to_device

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture
def pg():
    import async_copy_pipelined_gb300 as pg
    assert pg.device_status()[0] == 0
    yield pg
    pg.testing_f32_wide(-1)
    pg.testing_set_hooks(0, -1)
    pg.device_status()


def _sms():
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count


def _run(pg, A, B, M, N, K, stages=0, workspace="auto"):
    C = pg.gemm_f32(to_device(A, K), to_device(B, N), fill="tma", stages=stages, block_tile=128,
                    workspace=workspace)
    st, detail = pg.device_status()
    assert st == 0, f"device status {st} ({detail:#x})"
    return C.cpu().numpy()


# (M, N, K): wide rows = all rows (one round of 152 tiles on 152 SMs;
# ragged M, N and K), and some rows with the split 128 x 128 path below.
SHAPES = [(2432, 2048, 1024), (2400, 2000, 1030), (4096, 4096, 1024)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_wide_rows_equal_the_fma_chain(pg, M, N, K):
    sms = _sms()
    A, B = f32_operands("uniform", M, N, K, seed=71, fill="tma")
    want = oracle.gemm_fmaf_chain(A, B, M, N, K)
    plan = pg.plan_f32(M, N, K, lda=A.shape[1], ldb=B.shape[1], fill="tma", block_tile=128)
    assert plan["wide_rows"] == pg.f32_wide_rows(M, N, K, sms)
    if sms == 152:
        assert plan["wide_rows"] == (M if M < 4096 else 2432)
    for stages, ws in ((0, "auto"), (4, "auto"), (2, None)):
        assert_bitwise_equal(_run(pg, A, B, M, N, K, stages, ws), want, f"{M}x{N}x{K} S{stages} ws={ws}")
    pg.testing_f32_wide(0)
    assert pg.plan_f32(M, N, K, lda=A.shape[1], ldb=B.shape[1], fill="tma", block_tile=128)["wide_rows"] == 0
    assert_bitwise_equal(_run(pg, A, B, M, N, K), want, f"{M}x{N}x{K} without the wide kernel")


def test_forced_wide_rows_equal_the_fma_chain(pg):
    """Mode 1 takes a cut wherever one exists, here on a shape whose model
    keeps every row on 128 x 128 tiles."""
    M, N, K = 3000, 2048, 1024  # 24 strips of 8 wide tiles: 19 of them make one round
    sms = _sms()
    A, B = f32_operands("uniform", M, N, K, seed=72, fill="tma")
    pg.testing_f32_wide(1)
    rows = pg.plan_f32(M, N, K, lda=A.shape[1], ldb=B.shape[1], fill="tma", block_tile=128)["wide_rows"]
    assert rows == pg.f32_wide_rows(M, N, K, sms, mode=1)
    if sms == 152:
        assert rows == 2432
    assert_bitwise_equal(_run(pg, A, B, M, N, K), oracle.gemm_fmaf_chain(A, B, M, N, K), "forced wide rows")


def test_accumulating_calls_through_the_wide_kernel(pg):
    """K cut in two accumulating calls, each taking the wide kernel for all
    rows: the bits of one chain over the whole K."""
    import torch
    M, N, K = 2432, 2048, 2048
    A, B = f32_operands("uniform", M, N, K, seed=73, fill="tma")
    want = oracle.gemm_fmaf_chain(A, B, M, N, K)
    Ad, Bd = to_device(A, K), to_device(B, N)
    h = K // 2
    if _sms() == 152:
        assert pg.plan_f32(M, N, h, lda=A.shape[1], ldb=B.shape[1], fill="tma", block_tile=128)["wide_rows"] == M
    C = torch.full((M, N), float("nan"), device="cuda")
    pg.gemm_f32(Ad[:, :h], Bd[:h], C, fill="tma", block_tile=128)
    pg.gemm_f32(Ad[:, h:], Bd[h:], C, fill="tma", block_tile=128, accumulate=True)
    st, detail = pg.device_status()
    assert st == 0, f"device status {st} ({detail:#x})"
    assert_bitwise_equal(C.cpu().numpy(), want, "two accumulating calls")


@pytest.mark.parametrize("withhold", [0, 5])
def test_withheld_position_times_out_then_exact(pg, withhold):
    """A ring position the wide kernel never fills: its waits end with
    GEMM_ERR_TIMEOUT (family 6), and the next call is exact."""
    M, N, K = 2432, 2048, 1024
    A, B = f32_operands("uniform", M, N, K, seed=74, fill="tma")
    if pg.plan_f32(M, N, K, lda=A.shape[1], ldb=B.shape[1], fill="tma", block_tile=128)["wide_rows"] != M:
        pytest.skip("this device gives the shape no wide rows")
    pg.testing_set_hooks(10_000_000, withhold)
    pg.gemm_f32(to_device(A, K), to_device(B, N), fill="tma", block_tile=128)
    st, detail = pg.device_status()
    assert st == 6 and detail & 0xFF == 6 and (detail >> 8) & 0xFF in (1, 2), f"{st} {detail:#x}"
    pg.testing_set_hooks(0, -1)
    assert_bitwise_equal(_run(pg, A, B, M, N, K), oracle.gemm_fmaf_chain(A, B, M, N, K), "after timeout")


def test_host_buffers_through_the_wide_kernel(pg):
    """The host-buffer executor's K steps and row chunks on a shape whose
    chunk calls take the wide kernel: the bits of the device path."""
    import torch
    M, N, K = 2432, 2048, 4096
    A, B = (np.ascontiguousarray(x) for x in f32_operands("uniform", M, N, K, seed=75))
    want = oracle.gemm_fmaf_chain(A, B, M, N, K)
    got = pg.gemm_f32(torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory(), fill="tma")
    assert_bitwise_equal(got.numpy(), want, "host buffers")
