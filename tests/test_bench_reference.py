"""The benchmark's host-side parts, without a GPU: the reference arm (the CPU oracle timed on
the host cores), run as the driver runs it (one JSON line with the base contract's keys, on the
same metric, unit and workload as the GPU arm; ranks other than 0 exit without work), and the
parsing of the clock samples taken during the timed region."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra):
    env = dict(os.environ)
    env.update(env_extra)
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return [ln for ln in r.stdout.splitlines() if ln.startswith("{")]


def test_reference_arm_line():
    sys.path.insert(0, ROOT)
    import bench

    lines = _run({"RANK": "0"})
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["vs_baseline"] is None
    assert d["steps"] == 1 and d["warmup"] == 0 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"].startswith(bench.DEFAULT_WORKLOAD)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert cb["cores"] >= 1 and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_do_nothing():
    assert _run({"RANK": "1"}) == []


def test_clock_samples_parse(tmp_path):
    """The timed region's nvidia-smi samples: median SM clock, maximum clock, the throttle
    reasons seen at least once, and the median board power."""
    sys.path.insert(0, ROOT)
    import bench

    f = tmp_path / "clocks.csv"
    f.write_text("0, 1650, 2070, 1380.5, 0x4, Not Active, Not Active, Not Active, Active\n"
                 "0, 1700, 2070, 1395.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
                 "0, 1600, 2070, [N/A], 0x4, Not Active, Not Active, Not Active, Active\n"
                 "garbage line\n")
    c = bench.ClockSampler.parse(str(f))
    assert c["sm_mhz"] == 1650 and c["sm_max_mhz"] == 2070 and c["samples"] == 3
    assert c["reasons"] == ["sw_power_cap"]
    assert c["power_w"] == (1380.5 + 1395.0) / 2
