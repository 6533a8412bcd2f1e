"""Host-side logic that needs no GPU: the host path's row chunking, the
bench's roofline peak arithmetic, its workload descriptions and the reader
of the committed DRAM-traffic summary."""
import pytest

import async_copy_pipelined_gb300 as pg
import bench
from async_copy_pipelined_gb300 import inputs


@pytest.mark.parametrize("M", [1, 127, 128, 511, 512, 1023, 1024, 2048, 2500, 3300, 4096, 9000, 65536])
def test_host_row_chunks_cover_rows_once(M):
    ch = pg.host_row_chunks(M)
    assert ch[0][0] == 0 and ch[-1][1] == M
    assert all(a[1] == b[0] and a[0] < a[1] for a, b in zip(ch, ch[1:]))
    assert all((r1 - r0) % 128 == 0 for r0, r1 in ch[:-1])  # whole 128-row tiles but the last
    assert len(ch) <= pg.HOST_CHUNKS_MAX
    if M >= 2 * pg.HOST_CHUNK_MIN_ROWS:
        assert len(ch) >= 2 and all(r1 - r0 >= pg.HOST_CHUNK_MIN_ROWS for r0, r1 in ch[:-1])


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
