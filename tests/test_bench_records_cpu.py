"""The bench's use of committed ncu records: per-kernel times come from a
launch list only when it was taken on the same library sources and workload,
and the shares it apportions add up.  CPU only."""
import importlib.util
import json
import os

import pytest

_spec = importlib.util.spec_from_file_location(
    "bench", os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "bench.py"))
bench = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(bench)


def _record(tmp_path, monkeypatch, sha, workload="gqa_64x2048"):
    rec = {"workload": workload, "library_sha256": sha, "source": "test",
           "kernels": {"a": {"avg_us": 30.0, "per_layer": 1}, "b": {"avg_us": 5.0, "per_layer": 2}}}
    p = tmp_path / "decode_launches.json"
    p.write_text(json.dumps(rec))
    monkeypatch.setitem(bench.LAUNCH_RECORDS, "decode", str(p))


def test_breakdown_matches_sources(tmp_path, monkeypatch):
    _record(tmp_path, monkeypatch, bench.library_sha())
    out = bench.kernel_breakdown("decode", "gqa_64x2048", 32, 32 * 0.08)
    ks = out["kernels"]
    assert ks["a"]["share"] == pytest.approx(0.75) and ks["b"]["share"] == pytest.approx(0.25)
    assert sum(k["apportioned_live_us_per_layer"] for k in ks.values()) == pytest.approx(80.0, abs=1e-2)
    assert out["ncu_sum_per_layer_us"] == pytest.approx(40.0)


@pytest.mark.parametrize("sha,workload", [("0" * 64, "gqa_64x2048"), (None, "mha_100_fp16")])
def test_breakdown_refuses_stale_records(tmp_path, monkeypatch, sha, workload):
    _record(tmp_path, monkeypatch, sha or bench.library_sha(), workload=workload)
    assert "unavailable" in bench.kernel_breakdown("decode", "gqa_64x2048", 32, 1.8)


def test_library_sha_covers_every_source():
    """Any change to a kernel, launcher or the C header changes the hash."""
    d = os.path.join(bench.ROOT, "paged_quantized_kv_kvq_gb300", "csrc")
    srcs = [f for f in os.listdir(d) if f.endswith((".cu", ".cuh", ".h"))]
    assert "kvq_decode_impl.cuh" in srcs and "kvq_append.cu" in srcs and "kvq_prefill_ws_impl.cuh" in srcs
    assert len(bench.library_sha()) == 64
