"""The reference arm of bench.py on CPU: the JSON line it prints carries every key of the
benchmark contract, with the oracle's own timing in value, cpu_baseline and e2e."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line_has_the_contract_keys():
    sys.path.insert(0, ROOT)
    import bench
    args = type("A", (), {"steps": 2, "warmup": 1, "workload": "tiny_f32", "ref_step_seconds": 0.2})()
    line = bench.bench_reference(args, 0, 1)
    json.dumps(line)                                   # one JSON line, plain types only
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["n_gpus"] == 1 and line["steps"] == 2 and line["warmup"] == 1
    assert line["value"] > 0 and line["higher_is_better"] is True and line["dtype"] == "f64"
    assert "workload" in line["config"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    # rank > 0 of a multi-rank reference run does no work
    assert bench.bench_reference(args, 1, 2) is None
