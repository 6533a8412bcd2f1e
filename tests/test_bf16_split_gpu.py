"""The BF16 TMA fill's K split of the last round of tiles (gemm_bf16_ws):
when the tile count is not a multiple of the SM count, the persistent CTAs
share the last round and one more as equal runs of 64-deep K blocks, a tile
cut between two CTAs being finished by the second from the first one's FP32
accumulators, read back into tensor memory.  The tensor cores then issue the
same MMAs on the same accumulator values as without the split, so the bits
must equal the unsplit kernel's and every other fill's, and the results the
oracle's within the float32-accumulation bound (small integers: exactly)."""
import ctypes

import numpy as np
import pytest

from async_copy_pipelined_gb300 import inputs
from gpu_util import bf16_operands, to_device

import oracle

pytestmark = pytest.mark.gpu

# (M, N, K): 256-row tiles 17 x 9 = 153 (one over a round), 15 x 20 = 300,
# 16 x 16 = 256; a ragged edge tile and a ragged K block; two K blocks only.
SHAPES = [(4352, 2304, 512), (3840, 5120, 1024), (4096, 4096, 640), (4300, 2250, 200), (4352, 2304, 128)]


def _run(A, B, M, N, K, fill="tma", block_m=256, stages=0, workspace="auto"):
    import torch
    import async_copy_pipelined_gb300 as pg
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    pg.gemm_bf16(to_device(A, K), to_device(B, N), C, fill=fill, stages=stages, block_m=block_m, workspace=workspace)
    st, detail = pg.device_status()
    assert st == 0, f"device status {st} ({detail:#x})"
    return C.cpu().numpy()


def _bound_ok(got, A, B, M, N, K, what):
    want = oracle.gemm_bf16_f64(A, B, M, N, K)
    Aa = np.abs(inputs.bf16_bits_to_f32(A[:, :K])).astype(np.float64)
    Ba = np.abs(inputs.bf16_bits_to_f32(B[:, :N])).astype(np.float64)
    excess = np.abs(got - want) - K * 2.0 ** -22 * (Aa @ Ba)
    assert np.all(excess <= 0), f"{what}: per-element bound exceeded by {excess.max()}"


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("block_m", [128, 256])
def test_split_equals_unsplit_and_other_fills(M, N, K, block_m):
    import torch
    import async_copy_pipelined_gb300 as pg
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    A, B = bf16_operands("normal", M, N, K, 81)
    plan = pg.plan_bf16(M, N, K, lda=A.shape[1], ldb=B.shape[1], fill="tma", block_m=block_m)
    tiles = -(-M // block_m) * -(-N // 256)
    splits = tiles > sms and tiles % sms != 0 and -(-K // 64) >= 2
    assert (plan["workspace_bytes"] > 0) == splits
    if splits:
        assert plan["workspace_bytes"] == sms * (block_m * 256 * 4 + 8)
    got = _run(A, B, M, N, K, block_m=block_m)
    ref = _run(A, B, M, N, K, block_m=block_m, workspace=None)
    np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32), err_msg="split vs unsplit")
    other = _run(A, B, M, N, K, fill="cpasync", block_m=block_m)
    np.testing.assert_array_equal(got.view(np.uint32), other.view(np.uint32), err_msg="TMA split vs cp.async")
    _bound_ok(got, A, B, M, N, K, f"split {M}x{N}x{K} T{block_m}")


@pytest.mark.parametrize("block_m", [128, 256])
def test_split_small_integers_exact(block_m):
    M, N, K = 4352, 2304, 512
    A, B = bf16_operands("smallint", M, N, K, 82)
    got = _run(A, B, M, N, K, block_m=block_m)
    Ai = inputs.bf16_bits_to_f32(A[:, :K]).astype(np.int64)
    Bi = inputs.bf16_bits_to_f32(B[:, :N]).astype(np.int64)
    np.testing.assert_array_equal(got, (Ai @ Bi).astype(np.float32))


def test_workspace_is_checked():
    import torch
    import async_copy_pipelined_gb300 as pg
    M, N, K = 4352, 2304, 512
    A, B = bf16_operands("normal", M, N, K, 83)
    Ad, Bd = to_device(A, K), to_device(B, N)
    need = pg.plan_bf16(M, N, K, lda=A.shape[1], ldb=B.shape[1], fill="tma", block_m=256)["workspace_bytes"]
    assert need > 0
    C = torch.empty((M, N), device="cuda")
    lib = pg.lib()
    h = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ws = torch.empty(need + 64, dtype=torch.uint8, device="cuda")
    args = (M, N, K, Ad.data_ptr(), Ad.stride(0), Bd.data_ptr(), Bd.stride(0), C.data_ptr(), N, 2, 0, 256)
    assert lib.gemm_bf16_ws(*args, ws.data_ptr(), need - 1, h) == 1
    assert lib.gemm_bf16_ws(*args, ws.data_ptr() + 4, need, h) == 2
    ws.fill_(0xAB)  # garbage in the workspace does not matter
    assert lib.gemm_bf16_ws(*args, ws.data_ptr(), need, h) == 0
    assert pg.device_status()[0] == 0
    ref = _run(A, B, M, N, K, workspace=None)
    np.testing.assert_array_equal(C.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    C.fill_(7.0)  # the same workspace again: the last call's flags must not count
    assert lib.gemm_bf16_ws(*args, ws.data_ptr(), need, h) == 0
    assert pg.device_status()[0] == 0
    np.testing.assert_array_equal(C.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    # the cp.async fill has nothing to split: the workspace is ignored
    assert pg.plan_bf16(M, N, K, lda=A.shape[1], ldb=B.shape[1], fill="cpasync", block_m=256)["workspace_bytes"] == 0


def test_handover_wait_times_out_then_exact():
    """Heads store their accumulators but never raise the flag: every tail's
    epilogue gives up after the limit and records the hand-over role (6) of
    the BF16 family (2); the MMA warp's wait for the loaded accumulators runs
    out too; the next call is exact."""
    import async_copy_pipelined_gb300 as pg
    M, N, K = 4352, 2304, 512
    A, B = bf16_operands("normal", M, N, K, 84)
    ref = _run(A, B, M, N, K, workspace=None)
    assert pg.device_status()[0] == 0
    pg.testing_set_hooks(10_000_000, -1)
    pg.lib().gemm_testing_withhold_handover(1)
    try:
        import torch
        C = torch.empty((M, N), device="cuda")
        pg.gemm_bf16(to_device(A, K), to_device(B, N), C, fill="tma", block_m=256, workspace="auto")
        st, detail = pg.device_status()
    finally:
        pg.lib().gemm_testing_withhold_handover(0)
        pg.testing_set_hooks(0, -1)
    assert st == 6 and detail & 0xFF == 2 and (detail >> 8) & 0xFF == 6, f"{st} {detail:#x}"
    got = _run(A, B, M, N, K)
    np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32))
