"""The cache-qualifier options ("cp.async" tile-op reference: the prefetch
size of its operand contract and the cache_policy call parameter) change
where bytes sit in L2, never which bytes are copied: every option on every
fill that takes it gives the default call's bits, on ragged shapes that
exercise the guarded 16-byte and 4-byte copy paths and TMA's zero fill."""
import pytest

from gpu_util import assert_bitwise_equal, bf16_operands, f32_operands, to_device

import oracle

pytestmark = pytest.mark.gpu

F32_OPTION_SETS = [("l2_prefetch_128b",), ("a_evict_first", "b_evict_last"), ("a_evict_last", "b_evict_last"),
                   ("l2_prefetch_128b", "a_evict_first", "b_evict_first")]


def _f32(A, B, M, N, K, fill, stages, tile, options=()):
    import torch
    import async_copy_pipelined_gb300 as pg
    C = pg.gemm_f32(to_device(A, K), to_device(B, N), fill=fill, stages=stages, block_tile=tile, options=options)
    st, detail = pg.device_status()
    assert st == 0, f"device status {st} ({detail:#x})"
    torch.cuda.synchronize()
    return C.cpu().numpy()


@pytest.mark.parametrize("opts", F32_OPTION_SETS)
@pytest.mark.parametrize("fill,stages,tile", [("cpasync", 3, 128), ("cpasync", 2, 64), ("cpasync_mbar", 4, 128),
                                              ("cpasync_mbar", 2, 32), ("cpasync_ws", 4, 128), ("cpasync_ws", 2, 64),
                                              ("tma", 4, 128), ("tma", 2, 64)])
@pytest.mark.parametrize("M,N,K,lda", [(300, 260, 200, 203), (129, 513, 97, 100)])
def test_f32_options_keep_bits(opts, fill, stages, tile, M, N, K, lda):
    if fill == "tma":
        opts = tuple(o for o in opts if o != "l2_prefetch_128b")
    # TMA needs 16-byte row pitches: f32_operands raises lda and ldb to the
    # next one (NaN padding) for that fill.
    A, B = f32_operands("uniform", M, N, K, seed=21, lda=lda, fill=fill)
    policy = any("evict" in o for o in opts)
    if policy and fill != "tma" and (A.shape[1] % 4 or B.shape[1] % 4):
        # 4-byte copies carry no cache policy: the request is refused and
        # nothing is launched.
        import async_copy_pipelined_gb300 as pg
        with pytest.raises(pg.GemmError) as e:
            _f32(A, B, M, N, K, fill, stages, tile, opts)
        assert e.value.status == 3
        return
    want = oracle.gemm_fmaf_chain(A, B, M, N, K)
    got = _f32(A, B, M, N, K, fill, stages, tile, opts)
    assert_bitwise_equal(got, want, f"{fill} S{stages} T{tile} {opts}")


@pytest.mark.parametrize("opts", [("l2_prefetch_128b",), ("a_evict_first", "b_evict_last"),
                                  ("l2_prefetch_128b", "a_evict_last", "b_evict_last")])
@pytest.mark.parametrize("fill,stages,block_m", [("tma", 4, 128), ("tma", 3, 256), ("cpasync", 4, 128),
                                                 ("cpasync", 3, 256)])
def test_bf16_options_keep_bits(opts, fill, stages, block_m):
    import torch
    import async_copy_pipelined_gb300 as pg
    if fill == "tma":
        opts = tuple(o for o in opts if o != "l2_prefetch_128b")
    M, N, K = 300, 600, 200
    A, B = bf16_operands("normal", M, N, K, seed=22)
    Ad, Bd = to_device(A, K), to_device(B, N)
    ref = pg.gemm_bf16(Ad, Bd, fill=fill, stages=stages, block_m=block_m)
    got = pg.gemm_bf16(Ad, Bd, fill=fill, stages=stages, block_m=block_m, options=opts)
    st, detail = pg.device_status()
    assert st == 0, f"device status {st} ({detail:#x})"
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int32), ref.view(torch.int32)), f"bf16 {fill} {opts}"
