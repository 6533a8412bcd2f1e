"""The C ABI without a GPU: the library loads, exports every function the
public header declares, and validates / plans requests on the host exactly as
documented (no compute call is made)."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

import async_copy_pipelined_gb300 as pg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pg.build()
    return pg.lib()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \t\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M):
            if m.group(1) not in ("if", "while", "for", "return", "sizeof"):
                names.add(m.group(1))
    return names


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("gemm_f32", "gemm_bf16", "gemm_f32_plan", "gemm_bf16_plan", "gemm_status_string",
              "gemm_device_status", "gemm_selftest_bounded_wait", "gemm_version"):
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    path = pg.library_path()
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = _declared_functions() - exported
    assert not missing, f"declared but not exported: {sorted(missing)}"
    for n in _declared_functions():
        assert hasattr(lib, n)


def test_build_targets_sm103a_only():
    """One -gencode, sm_103a: no other architecture, no PTX for JIT."""
    from async_copy_pipelined_gb300 import buildlib
    flags = " ".join(buildlib.NVCC_FLAGS)
    assert flags.count("-gencode") == 1
    assert "arch=compute_103a,code=sm_103a" in flags


def test_version_and_status_strings(lib):
    assert lib.gemm_version() == 10200  # 1.2.0
    for code in range(7):
        s = pg.status_string(code)
        assert s.startswith("GEMM_")
    assert "unknown" in pg.status_string(99)


def _plan(M, N, K, lda=None, ldb=None, ldc=None, fill=2, stages=0, tile=0, a=256, b=256, c=256):
    p = pg.GemmPlan()
    st = pg.lib().gemm_f32_plan(M, N, K, a, lda if lda is not None else max(K, 1), b,
                                ldb if ldb is not None else max(N, 1), c, ldc if ldc is not None else max(N, 1),
                                fill, stages, tile, ctypes.byref(p))
    return st, p.as_dict()


def test_plan_defaults_and_shapes(lib):
    # The TMA fill's 128 tile: 1024 tiles = 6 rounds of 152 (the SM count
    # when no device can be asked) + 112 leave a last round to split, done by
    # one persistent CTA per SM whose hand-over space is one 64 KiB
    # accumulator tile and an 8-byte flag per CTA.
    # Its default ring depth is two stages (four for every other ring fill
    # and tile).
    st, p = _plan(4096, 4096, 4096, fill=2)
    assert st == 0 and p["block_m"] == 128 and p["stages"] == 2 and p["threads"] == 288
    assert (p["grid_x"], p["grid_y"], p["k_slices"]) == (32, 32, 256)
    assert p["persistent_ctas"] == 152 and p["workspace_bytes"] == 152 * (65536 + 8)
    assert p["smem_bytes"] == 2 * 16384 + 16 * 2 + 64 + 1024
    st, p = _plan(4096, 4096, 4096, fill=2, stages=4)
    assert st == 0 and p["stages"] == 4 and p["smem_bytes"] == 4 * 16384 + 16 * 4 + 64 + 1024
    st, p = _plan(1024, 1024, 1024, fill=2)  # automatic 64 tile
    assert st == 0 and p["block_m"] == 64 and p["stages"] == 4
    st, p = _plan(152 * 128, 2 * 128, 256, fill=2)  # 304 tiles: whole rounds, nothing to split
    assert st == 0 and p["persistent_ctas"] == 0 and p["workspace_bytes"] == 0
    st, p = _plan(1024, 1024, 4096, fill=2, tile=128)  # 64 tiles: one round, fewer CTAs than SMs
    assert st == 0 and p["persistent_ctas"] == 0 and p["workspace_bytes"] == 0
    st, p = _plan(4096, 4096, 4096, fill=1)
    assert st == 0 and p["persistent_ctas"] == 0 and p["workspace_bytes"] == 0
    assert (p["grid_x"], p["grid_y"]) == (32, 32)
    st, p = _plan(1024, 1024, 1024, fill=1)
    assert st == 0 and p["block_m"] == 64 and p["threads"] == 256 and p["stages"] == 4
    assert (p["grid_x"], p["grid_y"]) == (16, 16)
    st, p = _plan(4096, 4096, 4096, fill=3, stages=4)
    assert st == 0 and p["threads"] == 256 and p["a_copy_bytes"] == 16
    assert p["smem_bytes"] == 4 * 16384 + 16 * 4 + 64 + 1024
    st, p = _plan(256, 256, 256, fill=0)
    assert st == 0 and p["stages"] == 1 and p["smem_bytes"] == 8192
    st, p = _plan(3000, 5000, 1000, lda=1003, fill=1, tile=64)
    assert st == 0 and (p["grid_x"], p["grid_y"]) == (79, 47)
    assert p["a_copy_bytes"] == 4 and p["b_copy_bytes"] == 16 and p["k_slices"] == 63
    st, p = _plan(3000, 5000, 1000, lda=1003, fill=1, tile=128)
    assert st == 0 and (p["grid_x"], p["grid_y"]) == (40, 24)
    st, p = _plan(32, 32, 65536, fill=2, tile=32)
    assert st == 0 and p["threads"] == 64 and (p["thread_m"], p["thread_n"]) == (8, 4)
    assert (p["grid_x"], p["grid_y"], p["k_slices"]) == (1, 1, 4096)
    st, p = _plan(32, 32, 65536, fill=1, tile=32)
    assert st == 0 and p["threads"] == 32 and p["smem_bytes"] == 4 * 4096
    # The lesson's shared-memory arithmetic: one 64x64x16 stage is 8 KiB.
    for s in (2, 3, 4, 5, 6):
        st, p = _plan(512, 512, 512, fill=1, stages=s, tile=64)
        assert st == 0 and p["smem_bytes"] == s * 8192


@pytest.mark.parametrize("kw,code", [
    (dict(M=-1, N=4, K=4), 1),
    (dict(M=4, N=4, K=4, lda=3), 1),
    (dict(M=4, N=4, K=4, ldb=3), 1),
    (dict(M=4, N=4, K=4, ldc=3), 1),
    (dict(M=4, N=4, K=4, fill=5), 1),
    (dict(M=4, N=4, K=4, fill=0, stages=2), 1),
    (dict(M=4, N=4, K=4, fill=1, stages=1), 1),
    (dict(M=4, N=4, K=4, fill=2, stages=7), 1),
    (dict(M=4, N=4, K=4, tile=16), 1),
    (dict(M=4, N=4, K=4, a=0), 1),
    (dict(M=4, N=4, K=4, c=0), 1),
    (dict(M=4, N=4, K=4, a=258), 2),
    (dict(M=4, N=4, K=5, lda=5, fill=2), 2),
    (dict(M=4, N=4, K=4, a=260, fill=2), 2),
    (dict(M=65535 * 128 + 1, N=4, K=4, tile=128), 1),
])
def test_plan_refusals(lib, kw, code):
    args = dict(M=4, N=4, K=4)
    args.update(kw)
    st, _ = _plan(**args)
    assert st == code


def test_plan_accepts_what_only_some_fills_accept(lib):
    # lda not a multiple of 4: fine for sync / cp.async (4-byte copies), refused by TMA.
    assert _plan(4, 4, 5, lda=5, fill=0)[0] == 0
    assert _plan(4, 4, 5, lda=5, fill=1)[0] == 0
    assert _plan(4, 4, 5, lda=5, fill=3)[0] == 0
    assert _plan(4, 4, 5, lda=5, fill=2)[0] == 2
    # Empty problems are valid; K == 0 allows null A / B.
    assert _plan(0, 4, 4)[0] == 0
    assert _plan(4, 4, 0, a=0, b=0)[0] == 0


def test_bf16_plan(lib):
    p = pg.GemmPlan()
    L = pg.lib()
    st = L.gemm_bf16_plan(8192, 8192, 8192, 256, 8192, 256, 8192, 256, 8192, 2, 0, 0, ctypes.byref(p))
    assert st == 0
    d = p.as_dict()
    # 1024 tiles of 256 x 256: the 256-row tile, three 64 KiB stages, eight
    # epilogue warps with a 4 KiB staging box each.
    assert (d["block_m"], d["block_n"], d["block_k"], d["stages"]) == (256, 256, 64, 3)
    assert d["smem_bytes"] == 3 * 65536 + 8 * 4096 + 2048 <= 227 * 1024 and d["k_slices"] == 128
    assert d["threads"] == (1 + 1 + 8) * 32 and d["a_copy_bytes"] == 32768
    assert (d["grid_x"], d["grid_y"]) == (1024, 1)
    # Four stages only fit the 128-row tile: asking for them picks it.
    st = L.gemm_bf16_plan(8192, 8192, 8192, 256, 8192, 256, 8192, 256, 8192, 2, 4, 0, ctypes.byref(p))
    d = p.as_dict()
    assert st == 0 and (d["block_m"], d["stages"], d["threads"]) == (128, 4, (1 + 1 + 4) * 32)
    assert d["smem_bytes"] == 4 * 49152 + 4 * 4096 + 2048 and d["a_copy_bytes"] == 16384
    assert L.gemm_bf16_plan(64, 64, 64, 256, 64, 256, 64, 256, 64, 0, 0, 0, ctypes.byref(p)) == 0
    d = p.as_dict()
    assert d["stages"] == 1 and d["threads"] == 672 and d["a_copy_bytes"] == 16
    assert L.gemm_bf16_plan(64, 64, 64, 256, 64, 256, 64, 256, 64, 0, 2, 0, ctypes.byref(p)) == 1
    assert L.gemm_bf16_plan(64, 64, 64, 256, 64, 256, 64, 256, 64, 1, 0, 0, ctypes.byref(p)) == 0
    assert p.as_dict()["stages"] == 4 and p.as_dict()["threads"] == 416
    assert L.gemm_bf16_plan(64, 64, 64, 256, 64, 256, 64, 256, 64, 3, 0, 0, ctypes.byref(p)) == 3
    assert L.gemm_bf16_plan(64, 64, 60, 256, 60, 256, 64, 256, 64, 2, 0, 0, ctypes.byref(p)) == 2
    assert L.gemm_bf16_plan(64, 64, 64, 258, 64, 256, 64, 256, 64, 2, 0, 0, ctypes.byref(p)) == 2
    assert L.gemm_bf16_plan(64, 64, 64, 256, 64, 256, 64, 256, 64, 2, 5, 0, ctypes.byref(p)) == 1


# Without a device the planner assumes 152 SMs.  Waves of 128-row tiles w1
# against waves of 256-row tiles w2: the 256-row tile when 2 w2 < 1.08 w1.
@pytest.mark.parametrize("M,N,fill,stages,block_m,want", [
    (8192, 8192, 2, 0, 0, (256, 3)),      # w1 = 14, w2 = 7
    (2304, 2304, 2, 0, 0, (256, 3)),      # 162 tiles in 2 waves against 81 in 1
    (2048, 2048, 2, 0, 0, (128, 4)),      # 128 tiles in 1 wave against 64 in 1
    (3584, 3584, 2, 0, 0, (128, 4)),      # 392 tiles in 3 waves against 196 in 2
    (1024, 8192, 2, 0, 0, (256, 3)),      # 256 tiles in 2 waves against 128 in 1
    (8192, 8192, 2, 2, 0, (256, 2)),
    (8192, 8192, 2, 4, 0, (128, 4)),      # four stages: only the 128-row tile holds them
    (8192, 8192, 1, 0, 0, (256, 3)),      # the cp.async fill follows the same rule
    (8192, 8192, 0, 0, 0, (256, 1)),      # and the register fill, with its one stage
    (8192, 8192, 2, 0, 128, (128, 4)),    # an explicit tile keeps its own default depth
    (64, 64, 2, 0, 256, (256, 3)),
    (64, 64, 0, 1, 256, (256, 1)),
])
def test_bf16_plan_tile_choice(lib, M, N, fill, stages, block_m, want):
    p = pg.GemmPlan()
    st = pg.lib().gemm_bf16_plan(M, N, 64, 256, 64, 256, N, 256, N, fill, stages, block_m, ctypes.byref(p))
    d = p.as_dict()
    assert st == 0 and (d["block_m"], d["stages"]) == want
    assert d["threads"] == ({2: 1, 1: 8, 0: 16}[fill] + 1 + 4 * (want[0] // 128)) * 32


@pytest.mark.parametrize("fill,stages,block_m", [(2, 4, 256), (1, 4, 256), (2, 0, 64), (2, 0, 192), (2, 0, 512)])
def test_bf16_plan_tile_refusals(lib, fill, stages, block_m):
    p = pg.GemmPlan()
    assert pg.lib().gemm_bf16_plan(256, 256, 64, 256, 64, 256, 256, 256, 256, fill, stages, block_m,
                                   ctypes.byref(p)) == 1



def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    """No silent fallback: with the library path pointing nowhere, the binding raises."""
    import importlib
    mod = importlib.import_module("async_copy_pipelined_gb300")
    monkeypatch.setattr(mod, "_lib", None)
    monkeypatch.setattr(mod, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        mod.lib()


def test_testing_hooks_validate_and_reset(lib):
    """The test hooks are host-side settings: limits below 1 ms and
    positions below -1 are refused, and the defaults can always be restored
    (no device is touched)."""
    assert lib.gemm_testing_set_hooks(999_999, -1) == 1
    assert lib.gemm_testing_set_hooks(0, -2) == 1
    assert lib.gemm_testing_set_hooks(10_000_000, 3) == 0
    assert lib.gemm_testing_set_hooks(0, -1) == 0
    assert "gemm_testing_set_hooks" in _declared_functions()


@pytest.mark.parametrize("fill,opts,ok", [
    ("cpasync", ("l2_prefetch_128b",), True),
    ("cpasync_mbar", ("l2_prefetch_128b", "a_evict_first", "b_evict_last"), True),
    ("tma", ("a_evict_last", "b_evict_last"), True),
    ("tma", ("l2_prefetch_128b",), False),       # a cp.async qualifier
    ("sync", ("a_evict_first",), False),         # plain loads take no policy
    ("cpasync", ("a_evict_first", "a_evict_last"), False),
    ("tma", ("b_evict_first", "b_evict_last"), False),
])
def test_cache_options_accepted_where_they_apply(lib, fill, opts, ok):
    """The cache-qualifier options of the "cp.async" tile-op reference
    (prefetch size, L2 cache policy) are accepted only by fills whose copies
    carry them, and the plan echoes them."""
    if ok:
        p = pg.plan_f32(256, 256, 256, fill=fill, stages=0 if fill == "sync" else 2, options=opts)
        assert p["options"] == sum(pg.OPTIONS[o] for o in opts)
    else:
        with pytest.raises(pg.GemmError) as e:
            pg.plan_f32(256, 256, 256, fill=fill, stages=0 if fill == "sync" else 2, options=opts)
        assert e.value.status == 1


def test_cache_options_bf16_and_unknown_bits(lib):
    p = pg.plan_bf16(256, 256, 256, fill="cpasync", options=("l2_prefetch_128b", "b_evict_last"))
    assert p["options"] == 0x100 | 0x1000
    assert pg.plan_bf16(256, 256, 256, fill="tma", options=("a_evict_first",))["options"] == 0x200
    for fill, opts in (("tma", ("l2_prefetch_128b",)), ("sync", ("b_evict_last",))):
        with pytest.raises(pg.GemmError):
            pg.plan_bf16(256, 256, 256, fill=fill, options=opts)
    plan = pg.GemmPlan()
    assert lib.gemm_f32_plan(64, 64, 64, 256, 64, 256, 64, 256, 64, 2 | 0x4000, 2, 0, ctypes.byref(plan)) == 1
    assert lib.gemm_f32_plan(64, 64, 64, 256, 64, 256, 64, 256, 64, 2 | 0x80, 2, 0, ctypes.byref(plan)) == 1


def test_accumulate_option_fp32_only(lib):
    """GEMM_OPT_ACCUMULATE: every FP32 fill takes it (alone or beside cache
    options) and the plan reports it; the BF16 path refuses it as
    unsupported."""
    for fill in ("sync", "cpasync", "tma", "cpasync_mbar", "cpasync_ws"):
        plan = pg.GemmPlan()
        code = pg.FILL[fill] | pg.OPT_ACCUMULATE
        assert lib.gemm_f32_plan(300, 200, 100, 256, 100, 256, 200, 256, 200, code, 0, 0, ctypes.byref(plan)) == 0
        assert plan.options == pg.OPT_ACCUMULATE
    # the kernels that start from C are built with plain copies only
    plan = pg.GemmPlan()
    for fill, opt in (("tma", 0x1000), ("cpasync", 0x100), ("cpasync_ws", 0x200), ("cpasync_mbar", 0x800)):
        assert lib.gemm_f32_plan(256, 256, 256, 256, 256, 256, 256, 256, 256,
                                 pg.FILL[fill] | opt | pg.OPT_ACCUMULATE, 4, 0, ctypes.byref(plan)) == 3
    for fill in ("tma", "cpasync", "sync"):
        assert lib.gemm_bf16_plan(256, 256, 256, 256, 256, 256, 256, 256, 256, pg.FILL[fill] | pg.OPT_ACCUMULATE, 0,
                                  0, ctypes.byref(plan)) == 3


def _pieces(lib, tiles, ctas, k, split):
    out = (ctypes.c_int * 5)()
    per_cta = []
    for c in range(ctas):
        ps, idx = [], 0
        while lib.gemm_testing_f32_piece(tiles, ctas, k, split, c, idx, out):
            ps.append(tuple(out))
            idx += 1
        per_cta.append(ps)
    return per_cta


@pytest.mark.parametrize("tiles,ctas,k", [(1024, 152, 256), (960, 152, 63), (153, 152, 2), (208, 152, 5),
                                          (305, 152, 7), (304, 152, 9), (100, 152, 16), (1, 1, 3),
                                          (7, 3, 1), (7, 3, 2), (29, 4, 17), (5000, 148, 300)])
@pytest.mark.parametrize("split", [0, 1])
def test_persistent_schedule_covers_every_slice_once_in_k_order(lib, tiles, ctas, k, split):
    """The persistent FP32 kernel's work schedule, computed by the library's
    own code on the host: every (tile, K slice) is computed exactly once; a
    tile computed in two pieces is cut at one slice, the first piece handing
    its accumulators to the CTA right after, whose last piece it is; and
    that CTA does at least as many slices before the hand-over as the
    producing CTA does up to it, so a hand-over is normally ready in time."""
    per_cta = _pieces(lib, tiles, ctas, k, split)
    seen = {}
    for c, ps in enumerate(per_cta):
        for (t, s0, s1, frm, to) in ps:
            assert 0 <= t < tiles and 0 <= s0 < s1 <= k
            for sl in range(s0, s1):
                assert (t, sl) not in seen, f"slice {sl} of tile {t} twice"
                seen[(t, sl)] = c
    assert len(seen) == tiles * k
    heads = {}
    for c, ps in enumerate(per_cta):
        tos = [i for i, p in enumerate(ps) if p[4]]
        frs = [i for i, p in enumerate(ps) if p[3]]
        assert len(tos) <= 1 and len(frs) <= 1
        if not split:
            assert not tos and not frs
        for i in tos:
            t, s0, s1 = ps[i][:3]
            assert s0 == 0 and s1 < k
            heads[t] = (c, s1, sum(p[2] - p[1] for p in ps[:i + 1]))
        for i in frs:
            assert i == len(ps) - 1, "a continued tile is a CTA's last piece"
    for c, ps in enumerate(per_cta):
        for i, (t, s0, s1, frm, to) in enumerate(ps):
            if frm:
                hc, hend, h_done_at = heads[t]
                assert hc == c - 1 and hend == s0 and s1 == k
                # slices this CTA computes before starting the tail, against
                # the slices the producing CTA computes up to its hand-over
                before = sum(p[2] - p[1] for p in ps[:i])
                assert before >= h_done_at, (before, h_done_at)
    if split and tiles > ctas and tiles % ctas and k >= 2:
        # balanced: every CTA's total slices within one of the mean
        totals = [sum(p[2] - p[1] for p in ps) for ps in per_cta]
        assert max(totals) - min(totals) <= 1


def test_cache_policy_refused_on_four_byte_copies(lib):
    """Rows that are not 16-byte aligned are copied 4 bytes at a time, and
    those copies take the prefetch size but no L2 policy."""
    p = pg.plan_f32(300, 260, 200, lda=203, fill="cpasync", stages=2, options=("l2_prefetch_128b",))
    assert p["a_copy_bytes"] == 4 and p["options"] == 0x100
    for fill in ("cpasync", "cpasync_mbar"):
        with pytest.raises(pg.GemmError) as e:
            pg.plan_f32(300, 260, 200, lda=203, fill=fill, stages=2, options=("a_evict_first",))
        assert e.value.status == 3
        with pytest.raises(pg.GemmError) as e:
            pg.plan_f32(129, 513, 97, lda=100, fill=fill, stages=2, options=("b_evict_last",))
        assert e.value.status == 3
    assert pg.plan_f32(128, 512, 96, lda=100, fill="cpasync", stages=2, options=("b_evict_last",))["options"] == 0x1000


def test_producer_warp_fill_plan(lib):
    """The producer-warp cp.async fill: eight consumer warps plus four producer
    warps on the 128 tile (one on the 64 and 32 tiles), two stages by
    default, 16-byte copies; refused for the tensor-core GEMM."""
    p = pg.plan_f32(4096, 4096, 4096, fill="cpasync_ws")
    assert p["threads"] == 384 and p["stages"] == 2 and p["a_copy_bytes"] == 16
    assert pg.plan_f32(1024, 1024, 1024, fill="cpasync_ws", stages=3)["threads"] == 288
    assert pg.plan_f32(32, 32, 65536, fill="cpasync_ws", block_tile=32)["threads"] == 64
    with pytest.raises(pg.GemmError) as e:
        pg.plan_bf16(256, 256, 256, fill="cpasync_ws")
    assert e.value.status == 3


def test_bf16_plan_split_workspace():
    """The BF16 TMA fill offers the K split of the last round where the
    persistent CTAs (152 without a device) leave a partial round and a tile
    has at least two K blocks: one block_m x 256 FP32 slot and an 8-byte
    flag per CTA.  Other fills, whole rounds and single-block K offer none."""
    for block_m in (128, 256):
        p = pg.plan_bf16(4352, 2304, 512, fill="tma", block_m=block_m)
        assert p["workspace_bytes"] == 152 * (block_m * 256 * 4 + 8)
        assert p["persistent_ctas"] == 152
        assert pg.plan_bf16(4352, 2304, 512, fill="cpasync", block_m=block_m)["workspace_bytes"] == 0
        assert pg.plan_bf16(4352, 2304, 512, fill="sync", block_m=block_m)["workspace_bytes"] == 0
        assert pg.plan_bf16(4352, 2304, 64, fill="tma", block_m=block_m)["workspace_bytes"] == 0  # one K block
    assert pg.plan_bf16(8192, 8192, 8192, fill="tma", block_m=256)["workspace_bytes"] == 152 * (256 * 256 * 4 + 8)
    # 19 x 8 = 152 tiles of 256 rows: one whole round, nothing to split
    assert pg.plan_bf16(19 * 256, 8 * 256, 512, fill="tma", block_m=256)["workspace_bytes"] == 0
