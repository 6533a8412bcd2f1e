"""The K-split calls in a captured CUDA graph.

A split call's ready flags carry a value fixed when the call is made; a
graph replays the call with that same value.  Each tail lowers the flag it
has read, so every flag is back at 0 when a call ends and a replay cannot
take an old flag for a new one.  Checked directly (the flag words after a
call) and by replaying captured calls on new inputs."""
import numpy as np
import pytest

from gpu_util import assert_bitwise_equal, bf16_operands, f32_operands, to_device

import oracle

pytestmark = pytest.mark.gpu


def test_flags_are_lowered_after_a_split_call():
    import torch
    import async_copy_pipelined_gb300 as pg
    M, N, K = 2048, 2560, 96
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    A, B = f32_operands("uniform", M, N, K, seed=95, fill="tma")
    need = pg.plan_f32(M, N, K, lda=A.shape[1], ldb=B.shape[1], fill="tma", block_tile=128)["workspace_bytes"]
    assert need == sms * (128 * 128 * 4 + 8)
    ws = torch.full((need,), 0x5A, dtype=torch.uint8, device="cuda")
    ws[sms * 128 * 128 * 4:] = 0
    C = pg.gemm_f32(to_device(A, K), to_device(B, N), fill="tma", stages=2, block_tile=128, workspace=ws)
    assert pg.device_status()[0] == 0
    flags = ws[sms * 128 * 128 * 4:].view(torch.int64)
    assert int((flags != 0).sum()) == 0
    assert_bitwise_equal(C.cpu().numpy(), oracle.gemm_fmaf_chain(A, B, M, N, K), "split call")
    # BF16 (opt-in split)
    M, N, K = 4352, 2304, 512
    Ab, Bb = bf16_operands("normal", M, N, K, 96)
    need = pg.plan_bf16(M, N, K, lda=Ab.shape[1], ldb=Bb.shape[1], fill="tma", block_m=256)["workspace_bytes"]
    slots = sms * 256 * 256 * 4
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    pg.gemm_bf16(to_device(Ab, K), to_device(Bb, N), fill="tma", block_m=256, workspace=ws)
    assert pg.device_status()[0] == 0
    assert int((ws[slots:].view(torch.int64) != 0).sum()) == 0


def test_split_calls_replay_in_a_cuda_graph():
    import torch
    import async_copy_pipelined_gb300 as pg
    M, N, K = 2048, 2560, 96
    A, B = f32_operands("uniform", M, N, K, seed=97, fill="tma")
    Ad, Bd = to_device(A, K), to_device(B, N)
    C = torch.empty((M, N), device="cuda")
    Mb, Nb, Kb = 4352, 2304, 512
    Ab, Bb = bf16_operands("normal", Mb, Nb, Kb, 98)
    Abd, Bbd = to_device(Ab, Kb), to_device(Bb, Nb)
    Cb = torch.empty((Mb, Nb), device="cuda")
    wsb = torch.empty(pg.plan_bf16(Mb, Nb, Kb, lda=Ab.shape[1], ldb=Bb.shape[1], fill="tma",
                                   block_m=256)["workspace_bytes"], dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # warm-up: per-context setup happens outside the capture
        pg.gemm_f32(Ad, Bd, C, fill="tma", stages=2, block_tile=128, stream=s)
        pg.gemm_bf16(Abd, Bbd, Cb, fill="tma", block_m=256, workspace=wsb, stream=s)
    s.synchronize()
    assert pg.device_status()[0] == 0
    ref_b = Cb.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pg.gemm_f32(Ad, Bd, C, fill="tma", stages=2, block_tile=128, stream=s)
        pg.gemm_bf16(Abd, Bbd, Cb, fill="tma", block_m=256, workspace=wsb, stream=s)
    for seed in (99, 100, 101):
        A2, _ = f32_operands("uniform", M, N, K, seed=seed, fill="tma")
        Ad.copy_(to_device(A2, K))
        C.fill_(float("nan"))
        Cb.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert pg.device_status()[0] == 0
        assert_bitwise_equal(C.cpu().numpy(), oracle.gemm_fmaf_chain(A2, B, M, N, K), f"graph replay, seed {seed}")
        np.testing.assert_array_equal(Cb.cpu().numpy().view(np.uint32), ref_b.cpu().numpy().view(np.uint32))
