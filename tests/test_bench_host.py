"""bench.py's host-side pieces that need no GPU: the oracle CPU baseline
(all cores, and the same sample on one core in a child process) and the
source hash that ties a committed DRAM-traffic summary to the kernel it was
measured on."""
import argparse
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
pytest.importorskip("torch")
import bench  # noqa: E402


def test_cpu_baseline_reports_all_cores_and_one_core():
    out = bench.cpu_baseline(argparse.Namespace(config="tiny"))
    assert out["kind"] == "oracle" and out["value"] > 0
    one = out["one_core"]
    assert one["cores"] == 1 and one["value"] is not None and one["value"] > 0


def test_traffic_summaries_name_the_current_sources():
    # a summary whose hash does not match the sources yields no traffic figure
    for summary, sources in (("step_dram_traffic.txt", ("decode_step.cu", "attn_tc.cuh")),
                             ("attn_stream_dram_traffic.txt", ("attn_stream.cu", "attn_tc.cuh"))):
        r = bench.traffic_note(summary, *sources)
        assert r is None or 0.9 < r < 1.1
    assert bench.source_hash("decode_step.cu") != bench.source_hash("decode_step.cu", "attn_tc.cuh")
