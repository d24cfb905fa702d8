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
