"""Host-side logic that needs no GPU: the host path's row chunking, the
bench's roofline peak arithmetic, its workload descriptions and the reader
of the committed DRAM-traffic summary."""
import pytest

import async_copy_pipelined_gb300 as pg
import bench
from async_copy_pipelined_gb300 import inputs


@pytest.mark.parametrize("N,sms", [(4096, 152), (384, 152), (100, 148), (8192, 152), (1, 1), (70000, 152)])
def test_bf16_host_chunk_rows_fill_the_sms(N, sms):
    """A BF16 host-path chunk holds at least HOST_CHUNK_WAVES waves of
    128 x 128 tiles, in whole 256-row steps."""
    rows = pg.host_chunk_rows(N, sms)
    tiles_n = -(-N // 128)
    assert rows % 256 == 0 and rows >= pg.HOST_CHUNK_MIN_ROWS
    assert rows // 128 * tiles_n >= pg.HOST_CHUNK_WAVES * sms
    ch = pg.host_row_chunks(3000, N, sms)
    assert ch[0][0] == 0 and ch[-1][1] == 3000 and all(a[1] == b[0] for a, b in zip(ch, ch[1:]))


SCHEDULE_SHAPES = [(4096, 4096, 4096), (4096, 4096, 1100), (1792, 4096, 2048), (4096, 4096, 2047), (300, 64, 2576),
                   (300, 64, 2600), (300, 64, 2900), (300, 64, 2832), (300, 64, 2831),
                   (3300, 384, 256), (9000, 4096, 513), (1, 1, 1), (2048, 256, 1023), (65536, 4096, 65536),
                   (1700, 384, 2100), (0, 64, 64), (64, 0, 64), (100, 100, 0), (70000, 70000, 3000),
                   (8192, 8192, 2560), (640, 4096, 2576)]


@pytest.mark.parametrize("M,N,K", SCHEDULE_SHAPES)
def test_f32_host_schedule_covers_k_and_rows_once(M, N, K):
    """The native executor's cut: K blocks cover [0, K) in order, every bound
    but K a multiple of 16 (so each block of A starts on a 16-byte boundary
    of its row); a K from 512 + 2048 + 16 on is cut, into a first block of
    512 (or, with no room for a middle block, one of 512 to 767), middle
    blocks of at most 2048, and a last block of 2048 to 2063, at most 16
    blocks in all; the last block's row chunks cover [0, M) in order, in
    multiples of 128 rows but the last, at most 64 of them."""
    kb, rb = pg.host_schedule_f32(M, N, K, 152)
    assert kb[0] == 0 and kb[-1] == K
    assert all(a < b for a, b in zip(kb, kb[1:])) or K == 0
    assert all(k % 16 == 0 for k in kb[:-1])
    if K >= 512 + 2048 + 16:
        assert 3 <= len(kb) <= 17 and 2048 <= K - kb[-2] < 2064
        assert kb[1] == 512 or (len(kb) == 3 and 512 <= kb[1] < 768)
        if len(kb) < 17:  # up to 16 blocks; past that the middle ones grow
            assert all(b - a <= 2048 for a, b in zip(kb[1:-2], kb[2:-1]))
    else:
        assert kb == [0, K]
    assert rb[0] == 0 and rb[-1] == M and len(rb) - 1 <= 64
    assert all(a < b for a, b in zip(rb, rb[1:])) or M == 0
    assert all(r % 128 == 0 for r in rb[1:-1])


def test_f32_host_schedule_rows_follow_waves():
    """At N = 4096 on 152 SMs one wave of 128 x 128 tiles is 5 tile rows
    (640 rows): the last chunk is one wave, the others about two, and the
    first is 19 tile rows (608 tiles, exactly four rounds of 152), the
    largest whole-round block of at most two usual chunks."""
    kb, rb = pg.host_schedule_f32(4096, 4096, 4096, 152)
    assert kb == [0, 512, 2048, 4096]
    assert rb == [0, 2432, 3456, 4096]
    assert pg.lib().gemm_testing_host_streams(0, -1, 0) == 0
    try:
        assert pg.host_schedule_f32(4096, 4096, 4096, 152)[1] == [0, 1152, 2304, 3456, 4096]
    finally:
        assert pg.lib().gemm_testing_host_streams(0, -1, -1) == 0
    # chunks between the first and the last differ by at most one tile row
    rb = pg.host_schedule_f32(8192, 8192, 8192, 152)[1]
    sizes = [b - a for a, b in zip(rb[:-2], rb[1:-1])]
    assert max(sizes) - min(sizes) <= 128 and rb[-1] - rb[-2] >= 384


def test_f32_host_policy_hook_and_scratch():
    import ctypes
    lib = pg.lib()
    assert lib.gemm_testing_host_policy(-1, 0, 0, 0, 0, 0) == 1
    assert lib.gemm_testing_host_policy(8, 0, 0, 0, 0, 0) == 1
    try:
        assert lib.gemm_testing_host_policy(16, 32, 48, 64, 1, 3) == 0
        kb, rb = pg.host_schedule_f32(700, 300, 200, 152)
        assert kb[:2] == [0, 16] and kb[-1] == 200 and 32 <= 200 - kb[-2] < 48 and len(kb) >= 5
        assert rb == [0, 256, 512, 700]
    finally:
        assert lib.gemm_testing_host_policy(0, 0, 0, 0, 0, 0) == 0
    assert pg.host_schedule_f32(4096, 4096, 4096, 152)[0] == [0, 512, 2048, 4096]
    need = ctypes.c_size_t()
    assert lib.gemm_f32_host_scratch(1000, 999, 1001, ctypes.byref(need)) == 0
    def up(x):
        return -(-x // 256) * 256
    a = up(1000 * 1004 * 4)
    b = up(a + 1001 * 1000 * 4)
    c = up(b + 1000 * 1000 * 4)
    sms = 152  # no device here: the planning SM count
    # device copies of A, B and C, then one hand-over space per GEMM stream (up to 3)
    assert need.value == c + 3 * up(sms * (128 * 128 * 4 + 8))
    assert lib.gemm_f32_host_scratch(-1, 1, 1, ctypes.byref(need)) == 1
    assert lib.gemm_testing_host_streams(4, 1, 1) == 1 and lib.gemm_testing_host_streams(1, 2, 1) == 1
    assert lib.gemm_testing_host_streams(0, -1, -1) == 0


def test_fp32_peak_is_sms_times_lanes_times_clock():
    # 152 SMs x 128 FP32 lanes x 2 flops per FMA x 2070 MHz
    assert bench.fp32_peak_tflops(152, 2070.0) == pytest.approx(80.54784)
    assert bench.fp32_peak_tflops(76, 1000.0) == pytest.approx(76 * 128 * 2 * 1e9 / 1e12)


@pytest.mark.parametrize("name", sorted(inputs.WORKLOADS))
def test_workload_config_names_sizes(name):
    w = inputs.WORKLOADS[name]
    cfg = bench.workload_config(name, w, {"fill": "tma"})
    assert (cfg["M"], cfg["N"], cfg["K"], cfg["lda"]) == (w["M"], w["N"], w["K"], w["lda"])
    assert cfg["fill"] == "tma" and "flushed" in cfg["l2"] and str(w["seed"]) in cfg["workload"]


def test_profiled_traffic_only_for_matching_sources(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.md").write_text(
        "# traffic\n\n- source_sha: 0123abcd\n"
        "- traffic_bytes_per_launch[f32_4096:tma/S4/T128]: 329889792\n"
        "- `traffic_bytes_per_launch[bf16_8192:tma/S4/T0]: 1242865152`\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_sources_sha", lambda: "0123abcd")
    assert bench.profiled_traffic("f32_4096:tma/S4/T128") == 329889792
    assert bench.profiled_traffic("bf16_8192:tma/S4/T0") == 1242865152  # key holds a colon
    assert bench.profiled_traffic("f32_4096:cpasync/S4/T128") is None
    monkeypatch.setattr(bench, "kernel_sources_sha", lambda: "ffffffff")  # sources changed since
    assert bench.profiled_traffic("f32_4096:tma/S4/T128") is None


def test_kernel_sources_sha_covers_every_source(tmp_path, monkeypatch):
    csrc = tmp_path / "async_copy_pipelined_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "a.cu").write_text("x")
    (csrc / "b.cuh").write_text("y")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h1 = bench.kernel_sources_sha()
    (csrc / "host_exec.cu").write_text("w")  # sequences calls only: not hashed
    assert bench.kernel_sources_sha() == h1
    (csrc / "b.cuh").write_text("z")
    assert bench.kernel_sources_sha() != h1


def test_aliased_output_is_refused():
    """Byte-range overlap of C with A or B (views of one buffer) is refused;
    disjoint views of the same buffer are accepted."""
    import torch
    buf = torch.zeros(4096)
    A = buf[:1024].view(32, 32)
    B = buf[1024:2048].view(32, 32)
    pg._refuse_aliased_output(buf[2048:3072].view(32, 32), A, B)  # disjoint: no error
    with pytest.raises(ValueError, match="overlaps A"):
        pg._refuse_aliased_output(A, A, B)
    with pytest.raises(ValueError, match="overlaps B"):
        pg._refuse_aliased_output(buf[1500:2524].view(32, 32), A, B)
    # A padded view (ld 40 > 32 columns) spans through its last row only.
    Ap = buf[:40 * 31 + 32].as_strided((32, 32), (40, 1))
    pg._refuse_aliased_output(buf[40 * 31 + 32: 40 * 31 + 32 + 1024].view(32, 32), Ap, B[:1, :1])


def test_host_call_refuses_aliased_output_before_touching_a_gpu():
    import torch
    A = torch.zeros((64, 64))
    B = torch.zeros((64, 64))
    with pytest.raises(ValueError, match="overlaps A"):
        pg.gemm_f32(A, B, A)
    with pytest.raises(ValueError, match="one device"):
        pg.gemm_f32(A, B.to("meta"))


def test_kernel_sources_sha_ignores_comments_but_not_code(tmp_path, monkeypatch):
    csrc = tmp_path / "async_copy_pipelined_gb300" / "csrc"
    csrc.mkdir(parents=True)
    f = csrc / "k.cu"
    f.write_text('// header\nint a = 1; /* block */ const char *s = "x // y";\n')
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h1 = bench.kernel_sources_sha()
    f.write_text('// another header\n\nint a = 1;   /* other */ const char *s = "x // y";\n')
    assert bench.kernel_sources_sha() == h1  # comments and whitespace only
    f.write_text('// header\nint a = 2; /* block */ const char *s = "x // y";\n')
    assert bench.kernel_sources_sha() != h1  # code
    f.write_text('// header\nint a = 1; /* block */ const char *s = "x // z";\n')
    assert bench.kernel_sources_sha() != h1  # text inside a string literal is code
