"""Error paths that need a device: capability gate, argument refusals that
reach the device, and the bounded-wait timeout (made to expire on purpose by
waiting on a barrier nothing arrives on, with a short limit; no trap, no
hang, and the context must stay usable afterwards)."""
import numpy as np
import pytest

from gpu_util import assert_bitwise_equal, f32_operands, run_f32

import oracle

pytestmark = pytest.mark.gpu


def test_device_is_sm103():
    import torch
    assert torch.cuda.get_device_capability() == (10, 3)


def test_bounded_wait_times_out_and_context_survives():
    import async_copy_pipelined_gb300 as pg
    assert pg.device_status()[0] == 0  # clean before
    assert pg.selftest_bounded_wait(20000) == 0  # 20 ms limit
    st, detail = pg.device_status()
    assert st == 6, f"expected GEMM_ERR_TIMEOUT, got {st}"
    assert detail & 0xFF == 3  # self-test family
    assert pg.device_status() == (0, 0)  # reading cleared it
    # The context is intact: a GEMM right after is still exact.
    M, N, K = 64, 64, 64
    A, B = f32_operands("uniform", M, N, K, seed=1)
    got, _ = run_f32(A, B, M, N, K, "tma", 2, 64)
    assert_bitwise_equal(got, oracle.gemm_fmaf_chain(A, B, M, N, K), "after timeout")


def test_refusals_enqueue_nothing():
    import torch
    import async_copy_pipelined_gb300 as pg
    A = torch.ones((64, 64), device="cuda")
    B = torch.ones((64, 64), device="cuda")
    C = torch.full((64, 64), 9.0, device="cuda")
    cases = [
        (dict(fill="sync", stages=2), 1),
        (dict(fill="cpasync", stages=7), 1),
        (dict(fill="tma", stages=1), 1),
        (dict(fill="tma", block_tile=96), 1),
        (dict(fill=6), 1),
    ]
    for kw, code in cases:
        with pytest.raises(pg.GemmError) as e:
            pg.gemm_f32(A, B, C, **kw)
        assert e.value.status == code, kw
    # Misaligned base for TMA: a view starting one float into the buffer.
    buf = torch.ones((64, 68), device="cuda")
    with pytest.raises(pg.GemmError) as e:
        pg.gemm_f32(buf[:, 1:65], B, C, fill="tma")
    assert e.value.status == 2
    # The same view is fine for the sync / cp.async fills (4-byte copies).
    out = pg.gemm_f32(buf[:, 1:65], B, fill="cpasync")
    assert torch.all(out == 64.0)
    # bf16 with the mbarrier-completed cp.async fill is not implemented; the
    # register-path fill has exactly one stage.
    Ab = torch.ones((64, 64), dtype=torch.bfloat16, device="cuda")
    lib = pg.lib()
    st = lib.gemm_bf16(64, 64, 64, Ab.data_ptr(), 64, Ab.data_ptr(), 64, C.data_ptr(), 64, 3, 0, 0, None)
    assert st == 3
    st = lib.gemm_bf16(64, 64, 64, Ab.data_ptr(), 64, Ab.data_ptr(), 64, C.data_ptr(), 64, 0, 2, 0, None)
    assert st == 1
    st = lib.gemm_bf16(64, 64, 64, Ab.data_ptr(), 64, Ab.data_ptr(), 64, C.data_ptr(), 64, 2, 6, 0, None)
    assert st == 1  # stages above what fits in shared memory
    torch.cuda.synchronize()
    assert torch.all(C == 9.0), "a refused call wrote C"
    assert pg.device_status()[0] == 0


def test_mixed_host_and_device_operands_are_refused():
    """The kernels take raw pointers, so a host tensor next to device ones
    would be read as device memory: the binding refuses the call before any
    launch, for both GEMMs and for an output on the wrong side."""
    import torch
    import async_copy_pipelined_gb300 as pg
    Ad = torch.ones((64, 32), device="cuda")
    Bd = torch.ones((32, 48), device="cuda")
    Ah, Bh = Ad.cpu(), Bd.cpu()
    with pytest.raises(ValueError, match="one device"):
        pg.gemm_f32(Ad, Bh)
    with pytest.raises(ValueError, match="one device"):
        pg.gemm_f32(Ad, Bd, torch.empty((64, 48)))
    with pytest.raises(ValueError, match="one device"):
        pg.gemm_f32(Ah, Bd)  # host call with a device B
    with pytest.raises(ValueError, match="one device"):
        pg.gemm_bf16(Ad.bfloat16(), Bh.bfloat16())
    torch.cuda.synchronize()
    assert pg.device_status()[0] == 0
    C = pg.gemm_f32(Ad, Bd)  # the context still works
    assert torch.equal(C, torch.full((64, 48), 32.0, device="cuda"))
