"""bench.py's output contract, checked on the CPU through the reference arm
(the fp64 oracle timed on the host cores): one JSON line with the keys every
benchmark line carries, and the reference arm's own markers."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"}


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "1"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert KEYS <= set(d)
    assert d["impl"] == "reference"
    assert d["warmup"] >= 3                      # at least three untimed warm-up steps
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["config"]["workload"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"]


def test_clock_samples_are_taken_from_the_timed_region():
    """The clock figures come from the nvidia-smi samples stamped inside the timed
    region; a throttle reason outside it is not reported, one inside it is."""
    import datetime
    sys.path.insert(0, ROOT)
    import bench
    c = bench.ClockSampler(0)
    c.proc = type("Stopped", (), {"terminate": lambda self: None,
                                  "wait": lambda self, timeout=None: None})()
    c.t_start = datetime.datetime(2026, 1, 2, 3, 4, 5, 100000)
    c.t_end = datetime.datetime(2026, 1, 2, 3, 4, 5, 400000)
    idle = "Not Active, Not Active, Not Active, Not Active"
    c.lines = [
        "2026/01/02 03:04:05.050, 0, 1100, 2070, 200.5, 0x0, Not Active, Active, Not Active, Not Active",
        "2026/01/02 03:04:05.150, 0, 2070, 2070, 1300.1, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/01/02 03:04:05.250, 0, 2040, 2070, 1350.1, 0x0, " + idle,
        "2026/01/02 03:04:05.450, 0, 1200, 2070, 300.1, 0x0, " + idle,
    ]
    clk = c.stop()
    assert clk["samples"] == 4 and clk["samples_in_timed_region"] == 2
    assert clk["sm_mhz"] == 2055.0 and clk["sm_max_mhz"] == 2070.0
    assert clk["reasons"] == ["sw_power_cap"]
    # a region shorter than the sampling interval falls back to every sample
    c.t_start = c.t_end = datetime.datetime(2026, 1, 2, 3, 4, 6)
    clk = c.stop()
    assert clk["samples_in_timed_region"] == 0 and clk["sm_mhz"] == (1200 + 2040) / 2
    assert clk["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
