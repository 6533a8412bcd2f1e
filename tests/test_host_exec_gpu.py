"""The native FP32 host-buffer executor (gemm_f32_host): A, B and C in host
memory, B's rows and A's columns copied in K blocks, each block's GEMM
continuing the FMA chains of the block before it, the last block in row
chunks copied out as they finish.  Every result must equal the oracle's FMA
chain bit for bit, as the device path's does."""
import ctypes

import numpy as np
import pytest

from gpu_util import assert_bitwise_equal, f32_operands

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture
def small_policy():
    """K blocks of 16 / 32 / at most 48 from K = 64 on, row chunks of 128
    and 256 rows: many blocks and chunks on shapes the oracle finishes fast."""
    import async_copy_pipelined_gb300 as pg
    assert pg.lib().gemm_testing_host_policy(16, 32, 48, 64, 1, 3) == 0
    yield pg
    assert pg.lib().gemm_testing_host_policy(0, 0, 0, 0, 0, 0) == 0


def _host(A, cols, pinned=True):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(A))
    return (t.pin_memory() if pinned else t)[:, :cols]


@pytest.mark.parametrize("M,N,K", [(3000, 4096, 3100), (2300, 4096, 2700), (3300, 4096, 256)])
def test_default_schedule_equals_the_fma_chain(M, N, K):
    import torch
    import async_copy_pipelined_gb300 as pg
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    kb, rb = pg.host_schedule_f32(M, N, K, sms)
    assert (len(kb) > 2) == (K >= 512 + 2048 + 16) and len(rb) > 2
    A, B = f32_operands("uniform", M, N, K, seed=71, fill="tma")
    want = oracle.gemm_fmaf_chain(A, B, M, N, K)
    for fill in ("tma", "cpasync"):
        C = pg.gemm_f32(_host(A, K), _host(B, N), fill=fill)
        assert not C.is_cuda
        assert_bitwise_equal(C.numpy(), want, f"host executor {fill} {M}x{N}x{K}")


@pytest.mark.parametrize("fill", ["sync", "cpasync", "tma", "cpasync_mbar", "cpasync_ws"])
@pytest.mark.parametrize("M,N,K", [(700, 300, 200), (701, 301, 203), (129, 65, 70)])
def test_many_blocks_and_chunks_every_fill(small_policy, fill, M, N, K):
    pg = small_policy
    import torch
    kb, rb = pg.host_schedule_f32(M, N, K, torch.cuda.get_device_properties(0).multi_processor_count)
    assert len(kb) >= 4 and len(rb) >= 2
    A, B = f32_operands("uniform", M, N, K, seed=72, fill="tma")
    C = pg.gemm_f32(_host(A, K), _host(B, N), fill=fill)
    assert_bitwise_equal(C.numpy(), oracle.gemm_fmaf_chain(A, B, M, N, K), f"{fill} {M}x{N}x{K}")


@pytest.mark.parametrize("streams,split", [(2, 1), (3, 0), (2, 0)])
@pytest.mark.parametrize("M,N,K", [(700, 300, 200), (900, 260, 40)])
def test_several_gemm_streams(small_policy, streams, split, M, N, K):
    """Row chunks spread over two or three GEMM streams (every K step per
    chunk), with and without the K split of the last round: same bits."""
    pg = small_policy
    lib = pg.lib()
    assert lib.gemm_testing_host_streams(streams, split, -1) == 0
    try:
        A, B = f32_operands("uniform", M, N, K, seed=76, fill="tma")
        want = oracle.gemm_fmaf_chain(A, B, M, N, K)
        for fill in ("tma", "cpasync_ws"):
            C = pg.gemm_f32(_host(A, K), _host(B, N), fill=fill)
            assert_bitwise_equal(C.numpy(), want, f"{streams} GEMM streams, split {split}, {fill}")
    finally:
        assert lib.gemm_testing_host_streams(0, -1, -1) == 0


@pytest.mark.parametrize("M,N,K", [(5, 3, 0), (1, 1, 1), (130, 7, 3), (129, 200, 17), (0, 5, 5), (5, 0, 5)])
def test_tiny_and_empty_shapes(M, N, K):
    import torch
    import async_copy_pipelined_gb300 as pg
    A = np.random.default_rng(78).uniform(-1, 1, size=(M, K)).astype(np.float32)
    B = np.random.default_rng(79).uniform(-1, 1, size=(K, N)).astype(np.float32)
    C = pg.gemm_f32(torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory(), fill="tma")
    assert tuple(C.shape) == (M, N)
    if M and N and K:
        assert_bitwise_equal(C.numpy(), oracle.gemm_fmaf_chain(A, B, M, N, K), f"host executor {M}x{N}x{K}")
    elif M and N:  # the empty sum: +0 everywhere
        assert np.all(C.numpy().view(np.uint32) == 0)


def test_strided_and_pageable_host_buffers(small_policy):
    """Host A and B with row pitches beyond their widths (2-D copies), a host
    C with ldc > N whose extra columns must keep their sentinel, and
    pageable (not page-locked) memory."""
    pg = small_policy
    import torch
    M, N, K = 515, 130, 150
    A = np.asarray(f32_operands("uniform", M, N, K, seed=73, lda=K + 9)[0])
    B = np.asarray(f32_operands("uniform", M, N, K, seed=73, ldb=N + 5)[1])
    want = oracle.gemm_fmaf_chain(A, B, M, N, K)
    for pinned in (True, False):
        Cbuf = torch.full((M, N + 7), 12345.0)
        if pinned:
            Cbuf = Cbuf.pin_memory()
        pg.gemm_f32(_host(A, K, pinned), _host(B, N, pinned), Cbuf[:, :N], fill="tma")
        full = Cbuf.numpy()
        assert_bitwise_equal(full[:, :N].copy(), want, f"strided host buffers, pinned={pinned}")
        assert np.all(full[:, N:] == 12345.0)


def test_back_to_back_calls_share_the_scratch():
    """Two calls through the C ABI on one scratch with no wait between them:
    the second starts only after the first is done on the GPU, so each
    result is its own."""
    import torch
    import async_copy_pipelined_gb300 as pg
    lib = pg.lib()
    M, N, K = 2100, 1000, 2200
    ins = [f32_operands("uniform", M, N, K, seed=s, fill="tma") for s in (74, 75)]
    need = ctypes.c_size_t()
    assert lib.gemm_f32_host_scratch(M, N, K, ctypes.byref(need)) == 0
    scratch = torch.empty(need.value, dtype=torch.uint8, device="cuda")
    h = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    outs, keep = [], []
    for A, B in ins:
        Ah, Bh = _host(A, K), _host(B, N)
        C = torch.empty((M, N)).pin_memory()
        keep += [Ah, Bh]
        st = lib.gemm_f32_host(M, N, K, Ah.data_ptr(), Ah.stride(0), Bh.data_ptr(), Bh.stride(0), C.data_ptr(), N,
                               pg.FILL["tma"], 0, 0, scratch.data_ptr(), need.value, None, h)
        assert st == 0, pg.status_string(st)
        outs.append(C)
    torch.cuda.current_stream().synchronize()
    assert pg.device_status()[0] == 0
    for (A, B), C in zip(ins, outs):
        assert_bitwise_equal(C.numpy(), oracle.gemm_fmaf_chain(A, B, M, N, K), "back-to-back host calls")


def test_refusals():
    import torch
    import async_copy_pipelined_gb300 as pg
    lib = pg.lib()
    M, N, K = 64, 64, 64
    A = torch.zeros((M, K)).pin_memory()
    C = torch.zeros((M, N)).pin_memory()
    need = ctypes.c_size_t()
    assert lib.gemm_f32_host_scratch(M, N, K, ctypes.byref(need)) == 0
    scratch = torch.empty(need.value + 256, dtype=torch.uint8, device="cuda")
    h = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = (M, N, K, A.data_ptr(), K, A.data_ptr(), N, C.data_ptr(), N)
    assert lib.gemm_f32_host(*args, 2 | pg.OPT_ACCUMULATE, 0, 0, scratch.data_ptr(), need.value, None, h) == 1
    assert lib.gemm_f32_host(*args, 2, 0, 0, scratch.data_ptr(), need.value - 1, None, h) == 1
    assert lib.gemm_f32_host(*args, 2, 0, 0, None, 0, None, h) == 1
    assert lib.gemm_f32_host(*args, 2, 0, 0, scratch.data_ptr() + 16, need.value, None, h) == 2
    assert lib.gemm_f32_host(*args, 9, 0, 0, scratch.data_ptr(), need.value, None, h) == 1
    assert lib.gemm_f32_host(M, N, K, A.data_ptr(), K - 1, A.data_ptr(), N, C.data_ptr(), N, 2, 0, 0,
                             scratch.data_ptr(), need.value, None, h) == 1  # lda < K
    torch.cuda.current_stream().synchronize()
    assert pg.device_status()[0] == 0


def test_status_out_reports_a_timeout_then_clears():
    """With a ring position withheld (test hook), the executor's own copy of
    the status word reports the timeout; the next call reports 0 and is
    exact."""
    import torch
    import async_copy_pipelined_gb300 as pg
    lib = pg.lib()
    M, N, K = 300, 260, 100
    A, B = f32_operands("uniform", M, N, K, seed=77, fill="tma")
    Ah, Bh = _host(A, K), _host(B, N)
    need = ctypes.c_size_t()
    assert lib.gemm_f32_host_scratch(M, N, K, ctypes.byref(need)) == 0
    scratch = torch.empty(need.value, dtype=torch.uint8, device="cuda")
    word = torch.full((1,), -1, dtype=torch.int32).pin_memory()
    h = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    C = torch.empty((M, N)).pin_memory()
    args = (M, N, K, Ah.data_ptr(), Ah.stride(0), Bh.data_ptr(), Bh.stride(0), C.data_ptr(), N, pg.FILL["tma"], 0,
            0, scratch.data_ptr(), need.value, word.data_ptr(), h)
    assert pg.device_status()[0] == 0
    pg.testing_set_hooks(10_000_000, 1)
    try:
        assert lib.gemm_f32_host(*args) == 0
        torch.cuda.current_stream().synchronize()
    finally:
        pg.testing_set_hooks(0, -1)
    detail = int(word[0]) & 0xFFFFFFFF
    assert detail & 0xFF == 1 and (detail >> 8) & 0xFF in (1, 2), f"{detail:#x}"
    assert pg.device_status()[0] == 0  # the executor cleared the word
    assert lib.gemm_f32_host(*args) == 0
    torch.cuda.current_stream().synchronize()
    assert int(word[0]) == 0
    assert_bitwise_equal(C.numpy(), oracle.gemm_fmaf_chain(A, B, M, N, K), "after a timed-out host call")
