"""Host-side helpers of bench.py (CPU only)."""
import json

import numpy as np

import bench
from mla_decode_attention_07_gb300 import workloads as W


def test_traffic_record_needs_matching_workload_and_source(tmp_path):
    sha = bench.kernel_code_sha(bench.DECODE_SRC)
    rec = {"workload": "b16_h128_l4096", "code_sha256": sha,
           "dram_bytes_per_launch_full_workload": 123.0}
    p = tmp_path / "t.json"
    p.write_text(json.dumps(rec))
    assert bench.traffic_per_launch("b16_h128_l4096", str(p)) == 123.0
    assert bench.traffic_per_launch("tiny", str(p)) is None          # other workload
    rec["code_sha256"] = "0" * 64
    p.write_text(json.dumps(rec))
    assert bench.traffic_per_launch("b16_h128_l4096", str(p)) is None  # kernel changed since
    assert bench.traffic_per_launch("b16_h128_l4096", str(tmp_path / "missing.json")) is None


def test_sparse_sets_rotate_queries_and_positions():
    w = W.SparseWorkload("t", batch=3, h_q=16, seqlen=500, topk=64, pool_pages=9, seed=11)
    si = w.make()
    sets = bench.sparse_sets(w, si, 3)
    assert len(sets) == 3
    assert sets[0][0] is si.base.q and sets[0][1] is si.indices
    for q, idx, cnt in sets[1:]:
        assert q.shape == si.base.q.shape and idx.shape == si.indices.shape
        assert list(cnt) == [64, 64, 64]
        assert not np.array_equal(idx, si.indices) and not np.array_equal(q, si.base.q)
        assert ((idx >= 0) & (idx < 500)).all()


def test_sparse_cpu_baseline_reports_its_sample():
    w = W.SparseWorkload("t", batch=2, h_q=16, seqlen=300, topk=64, pool_pages=7, seed=12)
    r = bench.sparse_cpu_baseline(w.make(), 0.2)
    assert r["kind"] == "oracle" and r["unit"] == "TFLOP/s" and r["value"] > 0
    assert r["cores"] >= 1 and "query rows" in r["sample"]
