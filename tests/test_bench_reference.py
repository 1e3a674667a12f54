"""The bench's reference arm on the CPU: the oracle timed on decode tokens, one
token per step, after the asked-for warm-up steps, in the JSON line's shape."""
import argparse

import bench


def test_reference_arm_times_the_asked_steps():
    args = argparse.Namespace(steps=2, warmup=3, ref_seconds=5.0)
    d = bench.run_reference(args, 0, 1)
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert abs(d["ms_per_step"] - 1e3 / d["value"]) <= 0.01 * d["ms_per_step"] + 0.01
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_runs_on_rank_zero_only():
    args = argparse.Namespace(steps=2, warmup=3, ref_seconds=5.0)
    assert bench.run_reference(args, 1, 2) is None
