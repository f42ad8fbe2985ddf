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
