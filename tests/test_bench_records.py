"""The bench line's roofline.traffic comes from a committed ncu capture (profiles/traffic.json) and is reported
only while the kernel's sources hash to the capture's digest.  These checks keep the committed records in step
with the sources, so that the headline line never loses its measured traffic silently."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

HEADLINE = "decode_attn_kernel<fused> workload 5 bf16"


def _records():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        return json.load(f)


def test_headline_traffic_record_matches_the_current_sources():
    rec = bench.committed_traffic(HEADLINE)
    assert rec is not None, "profiles/traffic.json holds no capture of the headline kernel for the current sources"
    # ncu's DRAM bytes of one launch against the bytes the launch must move: nothing skipped, nothing re-read
    assert 0.99 <= rec["dram_bytes_per_launch"] / rec["algorithmic_bytes_per_launch"] <= 1.05


def test_every_record_names_an_existing_summary_and_matches_the_sources():
    for key, rec in _records().items():
        assert os.path.exists(os.path.join(ROOT, rec["profile"])), key
        assert bench.committed_traffic(key) is not None, f"{key}: sources changed since the capture"


def test_headline_algorithmic_bytes_match_the_bench_formula():
    from decode_attention_self_gb300 import workloads as W

    sb = bench.step_bytes(W.make_workload(5))
    assert _records()[HEADLINE]["algorithmic_bytes_per_launch"] == sb["self"] + sb["cross"] + sb["append"]
