"""Host-side accounting of bench.py, on CPU: the roofline's algorithmic bytes and the rule
that keeps a stale DRAM-traffic figure out of the result line."""

import json

import bench
import nf3_moe_gb300 as hm


def test_algorithmic_bytes_are_the_checkpoint_bytes():
    """Bytes per expert = the codes and scales of W13 [2I, H] and W2 [H, I] in the logical
    layout (the NVFP4 global scales, 8 bytes, are not counted)."""
    H, I = bench.SHAPE["H"], bench.SHAPE["I"]
    for fmt in (hm.FMT_NVFP4, hm.FMT_MXFP4, hm.FMT_NF3):
        w13 = sum(hm._matrix_bytes(fmt, 2 * I, H))
        w2 = sum(hm._matrix_bytes(fmt, H, I))
        assert bench.W13_BYTES[fmt] == w13
        assert bench.BYTES_PER_EXPERT[fmt] == w13 + w2
    # NVFP4 at H=6144, I=2048 by hand: W13 4096 x (3072 + 384), W2 6144 x (1024 + 128)
    assert bench.BYTES_PER_EXPERT[hm.FMT_NVFP4] == 4096 * 3456 + 6144 * 1152


def test_touched_counts_each_expert_once():
    fmts = [hm.FMT_NVFP4] * 64 + [hm.FMT_NF3] * 192
    ids = [[0, 5, 64, 200], [5, 0, 64, 201]]
    total, w13, n = bench.touched(ids, fmts)
    assert n == 5
    assert total == 2 * bench.BYTES_PER_EXPERT[hm.FMT_NVFP4] + 3 * bench.BYTES_PER_EXPERT[hm.FMT_NF3]
    assert w13 == 2 * bench.W13_BYTES[hm.FMT_NVFP4] + 3 * bench.W13_BYTES[hm.FMT_NF3]


def test_traffic_figure_is_dropped_when_stale(tmp_path, monkeypatch):
    rec = {"M": 8, "dram_bytes_per_launch": 123, "how": "capture",
           "source_sha16": bench.sources_sha16(bench.STREAM_SOURCES)}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "stream_gemm_traffic.json").write_text(json.dumps(rec))
    for src in bench.STREAM_SOURCES:                       # the same sources, copied beside it
        dst = tmp_path / src
        dst.parent.mkdir(parents=True, exist_ok=True)
        dst.write_bytes(open(f"{bench.ROOT}/{src}", "rb").read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.stream_traffic(8) == (123, "capture")
    assert bench.stream_traffic(4)[0] is None                              # another workload
    (tmp_path / bench.STREAM_SOURCES[0]).write_bytes(b"// changed\n")
    got, why = bench.stream_traffic(8)
    assert got is None and "stale" in why                                  # the kernel changed
    (tmp_path / "profiles" / "stream_gemm_traffic.json").unlink()
    assert bench.stream_traffic(8)[0] is None

