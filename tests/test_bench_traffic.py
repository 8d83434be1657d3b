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


def _csv_row(lid, kernel, metric, unit, value):
    return ",".join(f'"{x}"' for x in (lid, "1", "python3", "127.0.0.1", kernel, "1", "7", "(320, 1, 1)",
                                        "(8, 1, 1)", "0", "10.3", "Command line profiler metrics",
                                        metric, unit, value))


def test_record_traffic_from_an_ncu_csv(tmp_path, monkeypatch):
    """--record-traffic: units converted, launches of one kernel averaged, the
    decode call's split and combine kernels summed, sources hashed."""
    hdr = ",".join(f'"{x}"' for x in ("ID", "Process ID", "Process Name", "Host Name", "Kernel Name",
                                       "Context", "Stream", "Block Size", "Grid Size", "Device", "CC",
                                       "Section Name", "Metric Name", "Metric Unit", "Metric Value"))
    fwd = "void unnamed>::fwd_bf16_kernel<128, 1, 0, 0>(CUtensorMap_st, AttnParams)"
    lines = ["==PROF== Connected", hdr,
             _csv_row(0, fwd, "dram__bytes_read.sum", "Mbyte", "2.5"),
             _csv_row(0, fwd, "dram__bytes_write.sum", "byte", "500"),
             _csv_row(0, fwd, "gpu__time_duration.sum", "us", "3"),
             _csv_row(1, fwd, "dram__bytes_read.sum", "Mbyte", "1.5"),
             _csv_row(1, fwd, "dram__bytes_write.sum", "byte", "300"),
             _csv_row(1, fwd, "gpu__time_duration.sum", "us", "1"),
             _csv_row(2, "void decode_split_tc_kernel<128>(x)", "dram__bytes_read.sum", "Gbyte", "1"),
             _csv_row(2, "void decode_split_tc_kernel<128>(x)", "dram__bytes_write.sum", "byte", "10"),
             _csv_row(3, "void decode_combine_kernel<128>(x)", "dram__bytes_read.sum", "byte", "20"),
             _csv_row(3, "void decode_combine_kernel<128>(x)", "dram__bytes_write.sum", "byte", "30"),
             _csv_row(4, "void some_other_kernel(x)", "dram__bytes_read.sum", "byte", "99")]
    csv_path = tmp_path / "ncu.csv"
    csv_path.write_text("\n".join(lines) + "\n")
    table = tmp_path / "t.json"
    table.write_text(json.dumps({"_note": "kept"}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(table))
    out = bench.record_traffic(str(csv_path), "wl")
    assert out["fwd"]["dram_bytes_read"] == 2_000_000 and out["fwd"]["dram_bytes_write"] == 400
    assert out["fwd"]["gpu_time_ns_under_ncu"] == 2000 and out["fwd"]["launches_averaged"] == 2
    assert out["decode"]["bytes_per_launch"] == 1_000_000_000 + 10 + 20 + 30
    assert set(out) == {"fwd", "decode"}
    saved = json.loads(table.read_text())
    assert saved["_note"] == "kept" and saved["wl"] == out
    assert bench.ncu_traffic("wl", "fwd") == 2_000_400
    assert out["fwd"]["sources_sha256_16"]["fa_fwd_bf16.cu"] == bench.source_hash("fa_fwd_bf16.cu")
