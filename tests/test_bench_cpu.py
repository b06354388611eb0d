"""bench.py's host logic without a GPU: both arms print the same `config`, and the clock
summary covers the samples taken inside the timed region."""
import io
import json
import types
from contextlib import redirect_stdout

import bench


def test_reference_arm_prints_the_same_config(monkeypatch):
    monkeypatch.setattr(bench, "oracle_step_rate", lambda name, budget_s, threads: (1.0, "stub", 0.1, 1))
    args = types.SimpleNamespace(workload="cfg4", ref_budget=0.1, steps=5, warmup=3)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args, 0, 1)
    line = json.loads(buf.getvalue())
    assert line["impl"] == "reference"
    assert line["config"] == bench.config_of("cfg4", 1)
    assert line["config"]["packed_kv_bytes"] == 64 * 65536 * 8 * 100   # 3-bit: 32 * 3 + 4 bytes per token-head
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_clock_summary_counts_the_timed_window_only():
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.source, s.max_mhz, s.window = "test", 2070.0, (10.0, 10.02)
    s.rows = [(9.9, 1500.0, 300.0, 0x1), (10.005, 2070.0, 900.0, 0x0), (10.015, 2055.0, 950.0, 0x4),
              (10.5, 1200.0, 200.0, 0x20)]
    out = s.summary()
    assert out["samples"] == 2 and out["sm_mhz"] == (2070.0 + 2055.0) / 2
    assert out["reasons"] == ["sw_power_cap"] and out["sm_max_mhz"] == 2070.0
    assert out["whole_run"]["samples"] == 4 and "sw_thermal_slowdown" in out["whole_run"]["reasons"]
