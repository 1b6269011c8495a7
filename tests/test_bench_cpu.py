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


def test_traffic_figure_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    """The roofline's DRAM traffic comes from a committed ncu capture keyed by a hash of the
    kernel's sources: it is reported while they are unchanged and null once any of them changes."""
    sys.path.insert(0, ROOT)
    import bench
    srcs = bench.KERNEL_SOURCES["fwd_tc2_kernel"]
    got = bench.ncu_traffic("fwd_tc2_kernel", "mixtral_bf16", srcs)
    assert got is not None and got > 0                      # the committed capture is of these sources
    assert bench.ncu_traffic("fwd_tc2_kernel", "deepseek_bf16", srcs) is None   # no capture of that pairing
    # a changed source file: copy the sources into a scratch root, edit one, hash again
    for f in srcs:
        dst = tmp_path / f
        dst.parent.mkdir(parents=True, exist_ok=True)
        dst.write_bytes(open(os.path.join(ROOT, f), "rb").read())
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_bytes(open(os.path.join(ROOT, "profiles", "traffic.json"), "rb").read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.ncu_traffic("fwd_tc2_kernel", "mixtral_bf16", srcs) == got
    with open(tmp_path / srcs[0], "a") as fh:
        fh.write("\n// edited\n")
    assert bench.ncu_traffic("fwd_tc2_kernel", "mixtral_bf16", srcs) is None


def test_clock_samples_give_the_median_clock_and_the_active_reasons():
    """The clocks object of the JSON line from nvidia-smi samples taken during the timed region:
    median SM clock, highest max clock, every throttle reason seen active; malformed lines skipped."""
    sys.path.insert(0, ROOT)
    import bench

    class FakeProc:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0
    cs = bench.ClockSampler(0)
    cs.proc = FakeProc()
    cs.lines = ["1560, 2070, 1390.1, 0x4, Not Active, Not Active, Not Active, Active",
                "1575, 2070, 1395.0, 0x4, Not Active, Not Active, Not Active, Active",
                "1590, 2070, 1380.2, 0x0, Not Active, Not Active, Not Active, Not Active",
                "[N/A], 2070, 10.0, 0x0, Not Active, Not Active, Not Active, Not Active",   # no clock: skipped
                "garbage"]
    got = cs.stop()
    assert got == {"sm_mhz": 1575.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    cs.lines = ["1200, 2070, 700.0, 0x60, Active, Active, Not Active, Not Active"]
    assert cs.stop()["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]
    assert bench.ClockSampler(0).stop()["reasons"] == ["nvidia-smi unavailable"]   # never started


def test_issued_rows_follow_the_padded_work_model():
    """W_pad of the pages' padded-work model (rows rounded up to whole T_M-row tiles), and the
    pair kernel's rule: 256-row tiles with a 128-row tile at a group end that needs no more."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    import rdot_inputs as ri
    rng = np.random.default_rng(5)
    gs = rng.integers(0, 700, size=40)
    gs[[3, 9]] = 0
    for tm in (128, 256):
        assert bench.issued_rows(gs, tm, False) == sum(-(-int(x) // tm) * tm for x in gs)
    want = 0
    for x in map(int, gs):
        tiles, left = 0, x
        while left > 0:                       # whole 256-row tiles, then the end tile
            tiles += 128 if left <= 128 else 256
            left -= 256
        want += tiles
    assert bench.issued_rows(gs, 256, True) == want
    mix = ri.config_group_sizes("mixtral_bf16")
    assert abs(bench.issued_rows(mix, 256, True) / mix.sum() - 1.0391) < 1e-4      # 3.9 % tile tails
    assert abs(bench.issued_rows(mix, 256, False) / mix.sum() - 1.0781) < 1e-4
