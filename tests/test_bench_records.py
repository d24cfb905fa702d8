"""bench.py's lookup of the committed ncu traffic records (CPU only): every
key form resolves to its kernel's source file, and a record is used exactly
when its source hash matches the sources as they stand."""

import importlib.util
import json
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_module", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_every_traffic_key_resolves_to_its_source_file():
    b = _bench()
    recs = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    assert recs
    for key, entry in recs.items():
        kernel_file = key.split("#")[0].split("@")[0]
        assert os.path.exists(os.path.join(ROOT, "attention_learnable_sinks_gb300", "csrc", kernel_file)), key
        fresh = entry["source_sha"] == b.kernel_source_sha(kernel_file)
        got = b.traffic_record(key)
        assert (got is not None) == fresh, key
        if got is not None:
            assert got["dram_bytes_per_launch"] == entry["dram_bytes_per_launch"]


def test_unknown_keys_have_no_record():
    b = _bench()
    assert b.traffic_record("bwd.cu@no_such_workload") is None
    assert b.traffic_record("no_such_file.cu") is None


def test_reference_arm_prints_one_contract_line():
    """bench.py --impl reference (the oracle on the host cores) runs without a
    GPU and prints one JSON line with the keys the benchmark contract names."""
    import subprocess
    import sys
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"].startswith("dense")
