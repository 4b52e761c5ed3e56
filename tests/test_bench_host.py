"""Host-side accounting of bench.py: the algorithmic byte counts behind the metric and the
roofline, the traffic record's scaling, and the L2 rule each workload's timing follows."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_decode_bytes_counts_each_region_once():
    # one request of 1000 tokens, 2 KV heads, 8 query heads: 680 INT2 tokens at 2 x (32 + 8) B,
    # 320 BF16 tokens at 2 x 256 B per KV head, then q and out at 4 B per element
    want = 2 * (680 * 80 + 320 * 512) + 8 * 128 * 8
    assert bench.decode_bytes([1000], 2, 8) == want
    # a request inside sink + window has no INT2 tokens
    assert bench.decode_bytes([300], 1, 4) == 300 * 512 + 4 * 128 * 8
    # requests add up
    assert bench.decode_bytes([1000, 300], 2, 8) == want + 2 * 300 * 512 + 8 * 128 * 8


def test_int2_kernel_bytes_is_the_paged_part_plus_rotated_queries():
    assert bench.int2_kernel_bytes([100000] * 32, 8, 64) == 32 * 8 * 99680 * 80 + 32 * 64 * 512
    assert bench.int2_kernel_bytes([320], 8, 64) == 64 * 512


@pytest.mark.parametrize("name,flushed", [("tiny", True), ("qwen3_4b", True), ("qwen3_8b", False),
                                           ("qwen3_32b", False), ("ragged_128k", False)])
def test_l2_rule_per_workload(name, flushed):
    cfg = synth.config(name)
    assert bench.l2_flush_needed(cfg, cfg.ctx) == flushed
    text = bench.workload_config(cfg, cfg.ctx)["l2"]
    assert text.startswith("L2 flushed") == flushed
    assert text.startswith("inputs larger than L2") == (not flushed)


def test_traffic_record_scales_with_int2_bytes_and_tracks_the_source():
    with open(os.path.join(ROOT, "profiles", "decode_mma_traffic.json")) as f:
        rec = json.load(f)
    # the second argument is the INT2 bytes of the launch being reported
    got = bench.profiled_traffic(rec["workload"], 2 * rec["int2_bytes_per_launch"])
    if rec["source_sha256_16"] == bench.kernel_source_hash():
        assert got == pytest.approx(2.0 * rec["dram_bytes_per_launch"])
    else:
        assert got is None
    assert bench.profiled_traffic("another workload", rec["int2_bytes_per_launch"]) is None
