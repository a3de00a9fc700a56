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


PEAKS = {"bf16_tflops": 1930.3, "bf16_tflops_sustained": 1729.1, "hbm_gbs": 6792.4}


def test_binding_roof_follows_the_arithmetic_intensity():
    import inputgen
    b = _bench()
    c1 = inputgen.config("causal_4x4096_h64kv8")
    c2 = inputgen.config("window128_4x4096_h64kv8")
    r1, roofs1 = b.roofline_of(c1.unmasked_flops(), c1.algorithmic_bytes(), 6e-4, PEAKS, "m")
    r2, roofs2 = b.roofline_of(c2.unmasked_flops(), c2.algorithmic_bytes(), 1.5e-4, PEAKS, "m")
    assert r1["bound"] == "tensor" and r1["unit"] == "TFLOP/s"
    assert r2["bound"] == "hbm" and r2["unit"] == "GB/s"
    # both roofs are always reported; the line's roofline is the binding one
    assert r2["frac"] == roofs2["hbm"]["frac"] and r1["frac"] == roofs1["tensor"]["frac"]
    assert abs(roofs2["hbm"]["achieved"] - c2.algorithmic_bytes() / 1.5e-4 / 1e9) < 1e-6
    # E4M3 inputs: QK^T at twice the bf16 rate, PV at the bf16 rate -> 4/3 of the bf16 roof
    r3, _ = b.roofline_of(c1.unmasked_flops(), c1.algorithmic_bytes(), 6e-4, PEAKS, "m", True)
    assert abs(r3["peak"] - 4.0 / 3.0 * PEAKS["bf16_tflops"]) < 1e-9


def test_parity_stats():
    import numpy as np
    b = _bench()
    ref = np.zeros((3, 4))
    out = ref.copy()
    out[1, 2] = 0.5
    st = b.parity_stats(out, np.array([0.0, 1e-4, 0.0]), ref, np.zeros(3))
    assert st["rows"] == 3 and st["out_max_abs"] == 0.5 and st["finite"]
    assert abs(st["out_mean_abs"] - 0.5 / 12) < 1e-15 and abs(st["lse_max_abs"] - 1e-4) < 1e-15


def test_reference_arm_reports_its_measured_step_time_and_the_same_config():
    import subprocess
    import sys
    import time
    import inputgen
    b = _bench()
    t0 = time.perf_counter()
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_1x256_h4kv1", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300)
    wall = time.perf_counter() - t0
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["config"] == json.loads(json.dumps(
        b.config_dict(inputgen.config("tiny_1x256_h4kv1"), 1)))
    # a measured time (at most the process's wall time), not an extrapolation
    assert 0 < line["ms_per_step"] <= wall * 1e3
    assert line["ms_per_full_workload_extrapolated"] > 0


def test_log_lookup_takes_the_last_matching_line_and_skips_broken_ones(tmp_path):
    b = _bench()
    log = tmp_path / "runs.jsonl"
    mk = lambda wl, seed, v, impl=None: dict(
        {"config": {"workload": wl, "seed": seed}, "n_gpus": 1, "value": v},
        **({"impl": impl} if impl else {}))
    lines = [json.dumps(mk("a", 0, 1.0)), '{"config": {"workload": "a", "se',  # cut short
             json.dumps(mk("a", 1, 2.0)), json.dumps(mk("a", 0, 3.0, "reference")),
             json.dumps(mk("a", 0, 4.0)), ""]
    log.write_text("\n".join(lines))
    got = b.logged_line(str(log), b.run_key("a", 0, "ours", 1))
    assert json.loads(got)["value"] == 4.0
    assert json.loads(b.logged_line(str(log), b.run_key("a", 0, "reference", 1)))["value"] == 3.0
    assert b.logged_line(str(log), b.run_key("a", 0, "ours", 2)) is None
    assert b.logged_line(str(log), b.run_key("b", 0, "ours", 1)) is None
    assert b.logged_line(str(tmp_path / "absent.jsonl"), b.run_key("a", 0, "ours", 1)) is None


def test_resume_prints_the_logged_line_without_running_again(tmp_path):
    import subprocess
    import sys
    log = tmp_path / "runs.jsonl"
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--workload", "tiny_1x256_h4kv1", "--steps", "1", "--warmup", "3",
           "--log", str(log), "--resume"]
    first = subprocess.run(cmd, capture_output=True, text=True, timeout=300)
    assert first.returncode == 0, first.stderr
    assert len(log.read_text().splitlines()) == 1
    again = subprocess.run(cmd, capture_output=True, text=True, timeout=300)
    assert again.returncode == 0, again.stderr
    assert again.stdout.strip().splitlines()[-1] == first.stdout.strip().splitlines()[-1]
    assert len(log.read_text().splitlines()) == 1  # nothing appended, nothing rerun
    other = subprocess.run(cmd + ["--seed", "1"], capture_output=True, text=True, timeout=300)
    assert other.returncode == 0, other.stderr
    assert json.loads(other.stdout.strip().splitlines()[-1])["config"]["seed"] == 1
    assert len(log.read_text().splitlines()) == 2


def test_oracle_sample_of_a_given_size():
    import inputgen
    b = _bench()
    keep = {}
    _, n, _, thr, fl = b.oracle_rate(inputgen.config("tiny_1x256_h4kv1"), 1.0, keep=keep, rows=300)
    assert n == 300 and keep["out"].shape == (300, 64) and keep["lse"].shape == (300,)
    assert thr >= 1 and fl > 0
