"""bench.py's host-side helpers (no GPU): the device-source hash that keys
committed ncu traffic, and the rule that traffic is reported only for the
sources it was measured on."""
import importlib.util
import json
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return b


def test_source_hash_distinguishes_kernels():
    b = _bench()
    hs = {b.kernel_source_hash(64), b.kernel_source_hash(128), b.kernel_source_hash(64, True),
          b.kernel_source_hash(64, False, True)}
    assert len(hs) == 4 and all(len(h) == 16 for h in hs)
    assert b.kernel_source_hash(64) == b.kernel_source_hash(64)


def test_traffic_only_for_matching_sources(tmp_path, monkeypatch):
    b = _bench()
    prof = tmp_path / "profiles"
    prof.mkdir()
    cur = b.kernel_source_hash(64)
    (prof / "ncu_traffic.json").write_text(json.dumps({
        "w_current": {"kernel_source_hash": cur, "dram_bytes_per_launch": 1234},
        "w_stale": {"kernel_source_hash": "0" * 16, "dram_bytes_per_launch": 99},
    }))
    monkeypatch.setattr(b, "ROOT", str(tmp_path))  # where ncu_traffic looks for profiles/
    monkeypatch.setattr(b, "kernel_source_hash", lambda *a, **k: cur)
    assert b.ncu_traffic("w_current") == 1234.0
    assert b.ncu_traffic("w_stale") is None
    assert b.ncu_traffic("w_missing") is None


def test_committed_traffic_entries_are_well_formed():
    d = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
    for name, e in d.items():
        assert e["dram_bytes_per_launch"] > 0 and len(e["kernel_source_hash"]) == 16, name
        assert "kernel" in e and "source" in e, name
