"""The wide-row planner on the host (no GPU): which top rows of a TMA call on
the 128 tile go to the 128 x 256 kernel, and how many launches a call makes.

The planner takes whole rounds of wide tiles on the SMs (strip counts that
are multiples of SMs / gcd(SMs, wide tiles per strip)) and keeps a cut only
where its measured round costs make the call at least 1 % shorter; the rows
below run on the 128 x 128 path with its K split of the last round."""
import math

import pytest


@pytest.fixture(scope="module")
def pg():
    import async_copy_pipelined_gb300 as pg
    pg.lib()
    return pg


@pytest.mark.parametrize("M,N,K,rows", [
    (4096, 4096, 4096, 2432),   # 19 strips of 16 wide tiles: two rounds; 13 strips below
    (4096, 4096, 1024, 2432),
    (8192, 8192, 8192, 7296),   # 57 strips of 32: twelve rounds
    (2432, 2048, 1024, 2432),   # one round: every row
    (2400, 2000, 1030, 2400),   # the same round with a ragged last strip, N and K
    (3000, 2048, 1024, 0),      # one round and 80 tiles left: slower than the split 128 x 128 path
    (3840, 5120, 1024, 0),      # 38 strips make a round, 30 exist
    (4096, 4096, 1000, 0),      # K below 1024
    (1024, 4096, 2048, 0),
    (100, 4096, 4096, 0),
])
def test_model_decisions(pg, M, N, K, rows):
    assert pg.f32_wide_rows(M, N, K, 152) == rows
    plan = pg.plan_f32(M, N, K, lda=(K + 3) // 4 * 4, ldb=(N + 3) // 4 * 4, fill="tma", block_tile=128)
    assert plan["wide_rows"] == rows  # no device here: the planner assumes 152 SMs


@pytest.mark.parametrize("sms", [132, 148, 152, 160])
@pytest.mark.parametrize("M,N,K", [(4096, 4096, 4096), (8192, 8192, 2048), (6000, 3000, 1500), (2432, 2048, 1024)])
def test_cuts_are_whole_rounds_of_wide_tiles(pg, sms, M, N, K):
    for mode in (-1, 1):
        r = pg.f32_wide_rows(M, N, K, sms, mode)
        if r == 0:
            continue
        strips = (M + 127) // 128 if r == M else r // 128
        assert r == M or r % 128 == 0
        assert strips * ((N + 255) // 256) % sms == 0
        assert strips % (sms // math.gcd(sms, (N + 255) // 256)) == 0


def test_mode_zero_and_options_turn_it_off(pg):
    assert pg.f32_wide_rows(4096, 4096, 4096, 152, mode=0) == 0
    plan = pg.plan_f32(4096, 4096, 4096, lda=4096, ldb=4096, fill="tma", block_tile=128,
                       options=("a_evict_last",))
    assert plan["wide_rows"] == 0
    for fill in ("sync", "cpasync", "cpasync_mbar", "cpasync_ws"):
        assert pg.plan_f32(4096, 4096, 4096, lda=4096, ldb=4096, fill=fill, block_tile=128)["wide_rows"] == 0
    assert pg.plan_f32(4096, 4096, 4096, lda=4096, ldb=4096, fill="tma", block_tile=64)["wide_rows"] == 0


def test_knob_and_invalid_arguments(pg):
    lib = pg.lib()
    assert lib.gemm_testing_f32_wide(2) == 1
    assert lib.gemm_testing_f32_wide(-2) == 1
    assert lib.gemm_testing_f32_wide(0) == 0
    try:
        assert pg.plan_f32(4096, 4096, 4096, lda=4096, ldb=4096, fill="tma", block_tile=128)["wide_rows"] == 0
    finally:
        assert lib.gemm_testing_f32_wide(-1) == 0
    assert lib.gemm_testing_f32_wide_rows(-1, 4096, 4096, 152, -1) == -1
    assert lib.gemm_testing_f32_wide_rows(4096, 4096, 4096, 0, -1) == -1
    assert lib.gemm_testing_f32_wide_rows(4096, 4096, 4096, 152, 3) == -1


def test_rows_below_keep_their_split(pg):
    """At 4096^3 the 13 strips below the wide rows are 416 tiles of 128 x 128:
    one whole round, then the split region, as the plan reports."""
    plan = pg.plan_f32(4096, 4096, 4096, lda=4096, ldb=4096, fill="tma", block_tile=128)
    assert plan["wide_rows"] == 2432
    assert plan["persistent_ctas"] == 152
    assert plan["workspace_bytes"] == 152 * (128 * 128 * 4 + 8)
    assert (plan["grid_x"], plan["grid_y"]) == (32, 32)  # the 128 x 128 tiles of the whole C


def test_launches_per_call(pg):
    import bench
    # wide kernel + one-tile kernel (one whole round below) + split region
    assert bench.f32_kernels_per_call(pg, 4096, 4096, 4096, 4096, 4096, "tma", 2, 128) == 3
    assert bench.f32_kernels_per_call(pg, 4096, 4096, 4096, 4096, 4096, "tma", 2, 128, workspace=None) == 2
    # the wide kernel alone
    assert bench.f32_kernels_per_call(pg, 2432, 2048, 1024, 1024, 2048, "tma", 2, 128) == 1
    # no wide rows: the 128 x 128 path as before
    assert bench.f32_kernels_per_call(pg, 3840, 5120, 1024, 1024, 5120, "tma", 2, 128) == 2
    assert bench.f32_kernels_per_call(pg, 4096, 4096, 4096, 4096, 4096, "cpasync", 2, 128) == 1
