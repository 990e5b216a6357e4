"""The benchmark reports recorded DRAM traffic only for the kernel sources and
launch configuration the counters were taken with (host logic, no GPU)."""
import json
import os

import pytest

import bench
import block_scaled_mxfp4_gb300 as mx


def test_recorded_traffic_matches_only_its_plan_and_sources(tmp_path, monkeypatch):
    plan = mx.mxfp4_plan_gemm(8192, 8192, 8192, 0, 152)
    rec = {"large": {"kernel": "gemm_mxf4_pair", "dram_bytes_read": 10.0, "dram_bytes_write": 5.0,
                     "sources_sha1": "a" * 40, "plan": bench.plan_key(plan)}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_sources_sha1", lambda names=bench.KERNEL_SOURCES: "a" * 40)
    assert bench.recorded_traffic("large", "gemm_mxf4_pair", plan) == 15.0
    assert bench.recorded_traffic("large", "gemm_mxf4_kernel", plan) is None        # other kernel
    other = mx.mxfp4_plan_gemm(8192, 8192, 8192, 2, 152)
    assert bench.plan_key(other) != bench.plan_key(plan)
    assert bench.recorded_traffic("large", "gemm_mxf4_pair", other) is None         # other launch
    assert bench.recorded_traffic("decode", "gemm_mxf4_kernel", plan) is None       # no record
    monkeypatch.setattr(bench, "kernel_sources_sha1", lambda names=bench.KERNEL_SOURCES: "b" * 40)
    assert bench.recorded_traffic("large", "gemm_mxf4_pair", plan) is None          # sources changed


def test_committed_records_name_existing_summaries():
    with open(os.path.join(os.path.dirname(bench.__file__), "profiles", "traffic.json")) as f:
        recs = json.load(f)
    for name, rec in recs.items():
        if name.startswith("_"):
            continue
        assert rec["dram_bytes_read"] > 0, name
        assert os.path.exists(os.path.join(os.path.dirname(bench.__file__), rec["summary"])), name
