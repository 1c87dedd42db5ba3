"""bench.py's accounting on CPU: the algorithmic operation counts behind the
TOPS figures, against sums written out by hand from the layer shapes, and the
rule that the committed DRAM figure is reported only for the source it was
measured on."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import seeded_inputs as si  # noqa: E402


def test_mlp_operation_counts():
    # forward and weight gradient for every layer, delta propagation for all but the first;
    # two operations per multiply-accumulate
    B = 8192
    fwd = B * (4 * 4096 * 4096 + 4096 * 1000)
    dgrad = B * (3 * 4096 * 4096 + 4096 * 1000)
    assert bench.algorithmic_ops(si.by_name(3)) == 2.0 * (2 * fwd + dgrad)
    assert abs(bench.algorithmic_ops(si.by_name(3)) / 1e12 - 3.225) < 0.001
    B = 256
    fwd = B * (784 * 1024 + 1024 * 1024 + 1024 * 1024 + 1024 * 10)
    dgrad = B * (1024 * 1024 + 1024 * 1024 + 1024 * 10)
    assert bench.algorithmic_ops(si.by_name(1)) == 2.0 * (2 * fwd + dgrad)
    B = 32
    assert bench.algorithmic_ops(si.by_name(0)) == 2.0 * (2 * B * (64 * 64 + 64 * 10) + B * 64 * 10)


def test_cnn_operation_count():
    # 32x32x3 -> conv 3->64 (stride 1, 32x32) -> conv 64->128 (stride 2, 16x16) ->
    # conv 128->256 (stride 2, 8x8) -> pooling -> fc 256->10; no delta into the input
    B = 128
    c1 = B * 32 * 32 * 64 * 9 * 3
    c2 = B * 16 * 16 * 128 * 9 * 64
    c3 = B * 8 * 8 * 256 * 9 * 128
    fc = B * 256 * 10
    want = 2.0 * (2 * (c1 + c2 + c3 + fc) + (c2 + c3) + fc)
    assert bench.algorithmic_ops(si.by_name(2)) == want
    assert abs(want / 1e9 - 29.9) < 0.1


def test_dfp16_operation_count():
    B = 2048
    assert bench.algorithmic_ops(si.by_name(4)) == 2.0 * (2 * 3 * B * 2048 * 2048 + 2 * B * 2048 * 2048)


def test_committed_traffic_only_for_its_source(tmp_path, monkeypatch):
    w = si.by_name(3)
    assert bench.gemm_traffic_per_launch(si.by_name(1)) is None      # another workload
    got = bench.gemm_traffic_per_launch(w)
    assert got is None or got > 0
    # a summary whose hash is not the current source's is ignored
    text = open(bench.TRAFFIC_PROFILE).read()
    stale = tmp_path / "stale.md"
    stale.write_text(text.replace("kernel_source_sha256_16: ", "kernel_source_sha256_16: 0"))
    monkeypatch.setattr(bench, "TRAFFIC_PROFILE", str(stale))
    assert bench.gemm_traffic_per_launch(w) is None


def test_job_throughput_counts_every_rank():
    assert bench.job_throughput(1000, 4, 2.0) == 2000.0
