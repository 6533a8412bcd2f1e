"""Limits: the largest row count the FP32 grid allows, byte offsets beyond
2^32, and a K long enough to wrap every barrier ring hundreds of times.

The operands are seeded small integers generated on the device (entries in
{-2..2}): every partial sum is an integer of magnitude at most 4K < 2^24, so
the products are exact in any order and sampled rows are compared with the
exact integer product.  One row past the FP32 grid limit is refused (CPU
test of the plan); these runs sit exactly at it."""
import numpy as np
import pytest

from gpu_util import sample_rows

import oracle

pytestmark = pytest.mark.gpu


def _smallint(shape, seed, dtype):
    import torch
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randint(-2, 3, shape, generator=g, device="cuda", dtype=torch.int8).to(dtype)


def _host(x):
    """A device tensor as the oracle's host array: float32, or bfloat16 bits."""
    import torch
    if x.dtype == torch.bfloat16:
        return np.ascontiguousarray(x.cpu().view(torch.int16).numpy().view(np.uint16))
    return np.ascontiguousarray(x.cpu().numpy())


def _oracle_rows(A, B, rows):
    """The oracle's float64 definition on the sampled rows (exact for these
    integers), rounded to float32."""
    import torch
    a, b = _host(A[torch.as_tensor(rows, device=A.device)]), _host(B)
    K, N = b.shape
    fn = oracle.gemm_bf16_f64 if A.dtype == torch.bfloat16 else oracle.gemm_f64
    return fn(a, b, len(rows), N, K).astype(np.float32)


@pytest.mark.parametrize("fill,stages", [("tma", 4), ("cpasync", 3), ("cpasync_mbar", 2), ("sync", 1)])
def test_f32_rows_at_the_grid_limit_with_64bit_offsets(fill, stages):
    """M = 65535 x 128 rows on the 128-row tile (gridDim.y = 65535) and
    K = 132: A holds 4.4 GB, so row offsets pass 2^32 bytes (from row
    8134408 on) and the K tail is a partial slice."""
    import torch
    import async_copy_pipelined_gb300 as pg
    M, N, K = 65535 * 128, 24, 132
    A = _smallint((M, K), 11, torch.float32)
    B = _smallint((K, N), 12, torch.float32)
    plan = pg.plan_f32(M, N, K, fill=fill, stages=stages, block_tile=128)
    if fill == "tma":
        # persistent: one CTA per SM walks the 65535 tiles (the last round
        # split between CTAs, 65535 not being a multiple of the SM count)
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        assert plan["persistent_ctas"] == sms and plan["workspace_bytes"] > 0
    else:
        assert plan["grid_y"] == 65535
    C = pg.gemm_f32(A, B, fill=fill, stages=stages, block_tile=128)
    assert pg.device_status()[0] == 0
    rows = np.unique(np.concatenate([sample_rows(M, 16, seed=13, tiles=(128,)),
                                     np.arange(M - 130, M), [M // 2, (1 << 32) // (4 * K) + 1]]))
    np.testing.assert_array_equal(C[torch.as_tensor(rows, device=C.device)].cpu().numpy(),
                                  _oracle_rows(A, B, rows))
    del A, C
    torch.cuda.empty_cache()


@pytest.mark.parametrize("fill,stages,block_m", [("tma", 4, 128), ("cpasync", 4, 128), ("sync", 1, 128),
                                                 ("tma", 3, 256)])
def test_bf16_rows_beyond_4gb_offsets(fill, stages, block_m):
    """M = 2^23 + 72 ragged rows, K = 256: A holds 4.3 GB of bfloat16 and C
    8.6 GB, so both the operand and the output offsets pass 2^32 bytes."""
    import torch
    import async_copy_pipelined_gb300 as pg
    M, N, K = (1 << 23) + 72, 256, 256
    A = _smallint((M, K), 21, torch.bfloat16)
    B = _smallint((K, N), 22, torch.bfloat16)
    C = pg.gemm_bf16(A, B, fill=fill, stages=stages, block_m=block_m)
    assert pg.device_status()[0] == 0
    rows = np.unique(np.concatenate([sample_rows(M, 16, seed=23, tiles=(128,)), np.arange(M - 140, M),
                                     [M // 2]]))
    np.testing.assert_array_equal(C[torch.as_tensor(rows, device=C.device)].cpu().numpy(),
                                  _oracle_rows(A, B, rows))
    del A, C
    torch.cuda.empty_cache()


@pytest.mark.parametrize("fill,stages,block_m", [("tma", 2, 128), ("tma", 3, 128), ("tma", 4, 128),
                                                 ("cpasync", 2, 128), ("cpasync", 4, 128), ("sync", 1, 128),
                                                 ("tma", 2, 256), ("tma", 3, 256), ("cpasync", 3, 256)])
def test_bf16_long_k_wraps_the_ring(fill, stages, block_m):
    """K = 65536: 1024 K blocks per tile through a ring of 1 to 4 stages,
    i.e. hundreds of phase flips of every barrier; two 128-row tile rows (or
    one 256-row tile row) and three tile columns (one ragged) on persistent
    CTAs."""
    import torch
    import async_copy_pipelined_gb300 as pg
    M, N, K = 256, 600, 65536
    A = _smallint((M, K), 31, torch.bfloat16)
    B = _smallint((K, N), 32, torch.bfloat16)
    C = pg.gemm_bf16(A, B, fill=fill, stages=stages, block_m=block_m)
    assert pg.device_status()[0] == 0
    np.testing.assert_array_equal(C.cpu().numpy(), _oracle_rows(A, B, np.arange(M)))
