"""Host-side pieces of bench.py: the sampled parity figures attached to every
measured line, and the guarded read of the committed DRAM-traffic figure."""
import json
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
from quantized_weight_gb300 import inputs  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


@pytest.mark.parametrize("bits,group,prefill", [(4, 64, False), (8, 64, False), (1, 128, False), (4, 64, True)])
def test_sampled_parity_reads_zero_on_the_oracle_and_sees_a_wrong_output(bits, group, prefill):
    w = inputs.Workload("t", 3, 256, 96, bits, group, prefill)
    d = inputs.make(w.M, w.N, w.K, bits, group, seed=5, prefill=prefill)
    x = d["x_bf16"] if prefill else d["x"]
    f = oracle.qmm_bf16x if prefill else oracle.qmm_f32x
    y = f(x, oracle.pack(d["codes"], bits), d["scales"], d["biases"], w.N, w.K, bits, group).astype(np.float32)
    p = bench.sampled_parity(w, d, y, nsample=400)
    assert p["rel_l2"] < 1e-6 and p["max_err_over_max_ref"] < 1e-6
    bad = y.copy()
    bad[:, 7] = -bad[:, 7]                      # one wrong column in every row
    q = bench.sampled_parity(w, d, bad, nsample=400)
    assert q["rel_l2"] > 1e-3


def test_traffic_figure_is_dropped_when_a_kernel_source_changes(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    rel = os.path.relpath(src, ROOT)
    rec = {"headline": {"bytes_per_launch": 1234, "sources": [rel],
                        "sources_sha256": bench.sources_sha256([rel])}}
    tj = tmp_path / "traffic.json"
    tj.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_JSON", str(tj))
    assert bench.traffic_from_profile() == 1234.0
    src.write_text("kernel v2\n")
    assert bench.traffic_from_profile() is None
    monkeypatch.setattr(bench, "TRAFFIC_JSON", str(tmp_path / "missing.json"))
    assert bench.traffic_from_profile() is None


def test_committed_traffic_record_names_existing_sources():
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        pytest.skip("no committed traffic record")
    rec = json.load(open(path))["headline"]
    for rel in rec["sources"]:
        assert os.path.exists(os.path.join(ROOT, rel)), rel
    assert rec["bytes_per_launch"] > 0
