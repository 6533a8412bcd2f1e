"""gemm_f32_noalloc: the FP32 GEMM for callers that cannot allocate device
memory (an allocator that needs a GEMM while serving a request, code on a
fixed memory budget, latency-bound code that must not call cudaMalloc or
cudaFree, which may synchronise the device).  Its split of the last round
of tiles hands accumulators over through an array that lives inside the
library rather than in a caller buffer.

Called through the C ABI and compared, bit for bit as every FP32 result here
is, with the existing gemm_f32 entry point on the same inputs, on two calls
in a row (the second on other inputs, so the array still holds the first
call's contents).  Kept in a file that pytest collects last; it passes both
on its own in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest

from gpu_util import assert_bitwise_equal, f32_operands, to_device

pytestmark = pytest.mark.gpu


def _call(fn, Ad, Bd, M, N, K):
    import torch
    import async_copy_pipelined_gb300 as pg
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    h = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = fn(M, N, K, Ad.data_ptr(), Ad.stride(0), Bd.data_ptr(), Bd.stride(0), C.data_ptr(), N,
            pg.FILL["tma"], 4, 128, h)
    assert st == 0, pg.status_string(st)
    status, detail = pg.device_status()
    assert status == 0, f"device status {status} ({detail:#x})"
    return C.cpu().numpy()


@pytest.mark.parametrize("M,N,K", [(2048, 2560, 512), (1999, 2571, 133)])
def test_noalloc_matches_gemm_f32_on_two_calls_in_a_row(M, N, K):
    import torch
    import async_copy_pipelined_gb300 as pg
    lib = pg.lib()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = pg.plan_f32(M, N, K, lda=(K + 3) // 4 * 4, ldb=(N + 3) // 4 * 4, fill="tma", stages=4, block_tile=128)
    assert plan["workspace_bytes"] == sms * (128 * 128 * 4 + 8), "the shape must exercise the split"
    for seed in (41, 42):  # the second call finds the first call's contents in the array
        A, B = f32_operands("uniform", M, N, K, seed=seed, fill="tma")
        Ad, Bd = to_device(A, K), to_device(B, N)
        want = _call(lib.gemm_f32, Ad, Bd, M, N, K)
        got = _call(lib.gemm_f32_noalloc, Ad, Bd, M, N, K)
        assert not np.isnan(got).any()
        assert_bitwise_equal(got, want, f"gemm_f32_noalloc {M}x{N}x{K} seed {seed}")
