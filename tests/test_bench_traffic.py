"""The benchmark's DRAM-traffic lookup (CPU).

`roofline.traffic` comes from the committed ncu summary only while every
source of the kernel is byte-for-byte the one that was profiled; otherwise
it is null.  This checks both directions on a copy of the summary.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_summary_entries_are_well_formed():
    with open(bench.TRAFFIC_FILE) as f:
        rec = json.load(f)
    for wl, kernels in rec.items():
        if wl.startswith("_"):
            continue
        for name, e in kernels.items():
            assert e["bytes_per_launch"] == e["dram_bytes_read"] + e["dram_bytes_write"]
            for src in e["sources_sha256_16"]:
                assert os.path.exists(os.path.join(ROOT, "exact_io_aware_36_gb300", "csrc", src))


def test_lookup_voided_by_a_changed_source(tmp_path, monkeypatch):
    with open(bench.TRAFFIC_FILE) as f:
        rec = json.load(f)
    src = "fa_bwd_bf16.cu"
    fake = {"wl": {"k": {"sources_sha256_16": {src: bench.source_hash(src)},
                         "dram_bytes_read": 3, "dram_bytes_write": 4, "bytes_per_launch": 7}}}
    p = tmp_path / "t.json"
    p.write_text(json.dumps(fake))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(p))
    assert bench.ncu_traffic("wl", "k") == 7
    assert bench.ncu_traffic("other", "k") is None
    fake["wl"]["k"]["sources_sha256_16"][src] = "0" * 16
    p.write_text(json.dumps(fake))
    assert bench.ncu_traffic("wl", "k") is None
    assert rec  # the committed summary itself parsed
