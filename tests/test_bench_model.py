"""The byte and flop model of bench.py against the compulsory-traffic
figures worked out by hand for the two workloads of the bench step, and the
rule that a recorded DRAM-traffic figure is used only while the kernel
source it was measured on is unchanged.  CPU only."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from lm_local_sequence_causal_b300 import synthetic as syn  # noqa: E402


def test_headwise_bytes_at_the_qkv_size():
    # N = 16384 tokens, C = 6144, G = 384 groups, W = 4, bf16 (2 bytes):
    # fwd reads x and w and writes y; bwd reads x, w, dy and writes dx, dw
    fb, bb, ff, bf = bench.algorithmic(syn.qkv_headwise())
    N, C, G, W = 16384, 6144, 384, 4
    assert fb == 2 * (2 * N * C + N * G * W) == 452_984_832
    assert bb == 2 * (3 * N * C + 2 * N * G * W) == 704_643_072
    assert ff == 2 * N * C * W and bf == 4 * N * C * W


def test_lowrank_bytes_at_the_qkv_size():
    # R = 16: fwd reads x, z, U and writes y; bwd reads x, z, U, dy and
    # writes dx, dz, dU (the filters never reach memory)
    fb, bb, ff, bf = bench.algorithmic(syn.qkv_lowrank())
    N, C, W, R = 16384, 6144, 4, 16
    assert fb == 2 * (2 * N * C + N * R + R * C * W) == 403_963_904
    assert bb == 2 * (3 * N * C + 2 * N * R + 2 * R * C * W) == 606_601_216
    assert ff == 2 * N * C * W * R + 2 * N * C * W


def test_step_bytes_and_launch_count():
    hw = bench.algorithmic(syn.qkv_headwise())
    lr = bench.algorithmic(syn.qkv_lowrank())
    assert hw[0] + hw[1] + lr[0] + lr[1] == 2_168_193_024
    # head-wise fwd, bwd; low-rank fwd; low-rank bwd = U image + main + reduction
    assert bench.Problem.LAUNCHES_PER_STEP == 6


def test_recorded_traffic_needs_the_measured_source(tmp_path, monkeypatch):
    rec = json.load(open(os.path.join(ROOT, "profiles", "dram_traffic.json")))
    for name in bench.KERNEL_SOURCES:
        e = rec[name]
        same = e["source_sha256_16"] == bench.source_hash(bench.KERNEL_SOURCES[name])
        assert bench.recorded_traffic(name) == (e["bytes_per_launch"] if same else None), name
    # a changed source disables the figure
    monkeypatch.setattr(bench, "source_hash", lambda path: "0" * 16)
    assert all(bench.recorded_traffic(n) is None for n in bench.KERNEL_SOURCES)


def _ncu_row(i, name, metric, value):
    return ",".join(f'"{v}"' for v in (
        i, "1", "python3", "127.0.0.1", name, "1", "7", "(256, 1, 1)", "(148, 1, 1)", "0",
        "10.3", "Command line profiler metrics", metric, "byte", value))


def test_record_traffic_sums_each_entry_points_launches(tmp_path):
    # two bench steps of the six launches; the low-rank backward is three
    # launches, each entry point's bytes are per call
    names = ["void hw_tma_kernel<4, 16, 0, 64>(int)", "void hw_tma_kernel<4, 16, 1, 64>(int)",
             "void lr_fwd_tc<4, 1, 1>(int)", "void lr_u_image<4, 1>(int)",
             "void lr_bwd_tc<4, 1>(int)", "lr_reduce_tc(const float *)"]
    rows = ['==PROF== Connected to process 1',
            '"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",'
            '"Block Size","Grid Size","Device","CC","Section Name","Metric Name",'
            '"Metric Unit","Metric Value"']
    i = 0
    for step in range(2):
        for k, n in enumerate(names):
            rows.append(_ncu_row(i, n, "dram__bytes_read.sum", 1000 * (k + 1) + step))
            rows.append(_ncu_row(i, n, "dram__bytes_write.sum", 10 * (k + 1)))
            i += 1
    csv_path = tmp_path / "launches.csv"
    csv_path.write_text("\n".join(rows) + "\n")
    out = bench.record_traffic(str(csv_path), "cmd", out_path=str(tmp_path / "t.json"))
    assert json.load(open(tmp_path / "t.json")) == out
    assert out["headwise_fwd"]["read"] == 1000 and out["headwise_fwd"]["write"] == 10
    assert out["headwise_bwd"]["bytes_per_launch"] == 2000 + 20
    assert out["lowrank_fwd"]["bytes_per_launch"] == 3000 + 30
    # 4000 + 5000 + 6000 read in the first step, one byte more per launch in the
    # second: 15001.5 per call, truncated; 40 + 50 + 60 written
    assert out["lowrank_bwd"]["read"] == 15001 and out["lowrank_bwd"]["write"] == 150
    for name in bench.KERNEL_SOURCES:
        assert out[name]["source_sha256_16"] == bench.source_hash(bench.KERNEL_SOURCES[name])
