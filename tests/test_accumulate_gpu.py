"""GEMM_OPT_ACCUMULATE (gemm_f32(accumulate=True)): each element's FMA chain
continues from the value C holds.  A call over the first K0 columns of A and
rows of B, then accumulating calls over the rest, must give the oracle's FMA
chain over all K bit for bit, on every fill, stage count and tile, with the
K split of the last round of tiles and without it, (the native host-buffer executor, which uses the option for its K steps,
is tested in test_host_exec_gpu.py)."""
import numpy as np
import pytest

from gpu_util import F32_VARIANTS, assert_bitwise_equal, f32_operands, to_device

import oracle

pytestmark = pytest.mark.gpu


def _gemm_in_k_pieces(A, B, M, N, K, cuts, fill, stages, tile, workspace="auto"):
    import torch
    import async_copy_pipelined_gb300 as pg
    Ad, Bd = to_device(A, K), to_device(B, N)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    bounds = [0] + list(cuts) + [K]
    for j, (k0, k1) in enumerate(zip(bounds, bounds[1:])):
        pg.gemm_f32(Ad[:, k0:k1], Bd[k0:k1], C, fill=fill, stages=0 if fill == "sync" else stages,
                    block_tile=tile, accumulate=j > 0, workspace=workspace)
    st, detail = pg.device_status()
    assert st == 0, f"device status {st} ({detail:#x})"
    return C.cpu().numpy()


@pytest.mark.parametrize("fill,stages,tile", F32_VARIANTS)
def test_k_pieces_equal_the_fma_chain(fill, stages, tile):
    """Ragged M and N, a ragged K tail in each piece, three pieces.  TMA
    needs 16-byte aligned column offsets into A, so its cuts are multiples
    of four floats; the other fills also take an odd cut (A and B then start
    on 4-byte boundaries and move in 4-byte copies)."""
    M, N, K = 173, 150, 97
    A, B = f32_operands("uniform", M, N, K, seed=61, fill="tma")
    want = oracle.gemm_fmaf_chain(A, B, M, N, K)
    cuts = (20, 52) if fill == "tma" else (19, 52)
    got = _gemm_in_k_pieces(A, B, M, N, K, cuts, fill, stages, tile)
    assert_bitwise_equal(got, want, f"{fill} S{stages} T{tile} cuts {cuts}")


@pytest.mark.parametrize("M,N,K,cuts", [(2048, 2560, 96, (48,)), (1999, 2571, 133, (32, 64)),
                                        (3840, 5120, 512, (256,))])
def test_k_pieces_through_the_split_schedule(M, N, K, cuts):
    """Shapes whose 128 x 128 tiles overrun whole rounds of SMs: each TMA
    call splits its last round in K (heads, whole tiles and tails of the
    persistent kernel), and with accumulate every piece that starts a tile
    starts from C."""
    import torch
    import async_copy_pipelined_gb300 as pg
    A, B = f32_operands("uniform", M, N, K, seed=62, fill="tma")
    want = oracle.gemm_fmaf_chain(A, B, M, N, K)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    k_first = cuts[0]
    plan = pg.plan_f32(M, N, k_first, lda=A.shape[1], ldb=B.shape[1], fill="tma", stages=4, block_tile=128)
    assert plan["persistent_ctas"] == sms, "the first piece must take the split path"
    for stages in (2, 4):
        got = _gemm_in_k_pieces(A, B, M, N, K, cuts, "tma", stages, 128)
        assert_bitwise_equal(got, want, f"{M}x{N}x{K} S{stages} split")
    got = _gemm_in_k_pieces(A, B, M, N, K, cuts, "tma", 4, 128, workspace=None)
    assert_bitwise_equal(got, want, f"{M}x{N}x{K} unsplit")


def test_accumulate_with_k_zero_leaves_c():
    import torch
    import async_copy_pipelined_gb300 as pg
    M, N = 130, 70
    C = torch.arange(M * N, dtype=torch.float32, device="cuda").reshape(M, N) * 0.5 - 7.0
    before = C.clone()
    A = torch.empty((M, 0), dtype=torch.float32, device="cuda")
    B = torch.empty((0, N), dtype=torch.float32, device="cuda")
    for fill in ("sync", "cpasync", "tma", "cpasync_mbar", "cpasync_ws"):
        pg.gemm_f32(A, B, C, fill=fill, accumulate=True)
    torch.cuda.synchronize()
    assert torch.equal(C.view(torch.int32), before.view(torch.int32))
    pg.gemm_f32(A, B, C, fill="tma")  # without accumulate: the empty sum
    torch.cuda.synchronize()
    assert torch.equal(C, torch.zeros_like(C))


def test_accumulate_from_arbitrary_c_matches_the_chain_from_that_value():
    """A C that no earlier call wrote: each element is C's value followed by
    one fma per k ascending, computed on the CPU with numpy's float32 fma
    emulated in float64 (exact for these small-integer operands)."""
    import torch
    import async_copy_pipelined_gb300 as pg
    M, N, K = 150, 136, 40
    rng = np.random.default_rng(63)
    A = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
    B = rng.integers(-4, 5, size=(K, N)).astype(np.float32)
    C0 = rng.integers(-1000, 1000, size=(M, N)).astype(np.float32)
    want = (C0.astype(np.float64) + A.astype(np.float64) @ B.astype(np.float64)).astype(np.float32)
    for fill in ("sync", "cpasync", "tma", "cpasync_mbar", "cpasync_ws"):
        C = torch.from_numpy(C0).cuda()
        pg.gemm_f32(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), C, fill=fill, accumulate=True)
        assert pg.device_status()[0] == 0
        assert_bitwise_equal(C.cpu().numpy(), want, f"{fill} from arbitrary C")


def test_accumulate_refusals():
    import torch
    import async_copy_pipelined_gb300 as pg
    A = torch.zeros((8, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        pg.gemm_f32(A, A.clone(), accumulate=True)  # no C to continue from
    with pytest.raises(ValueError):
        pg.gemm_f32(A.cpu(), A.cpu(), torch.zeros((8, 8)), accumulate=True)  # host tensors
