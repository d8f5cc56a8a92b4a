"""bench.py's reference arm runs on the host cores only, so its JSON line can be
checked here: one line, the contract's keys, and the numbers it derives."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny", "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, check=True, cwd=ROOT, timeout=600)
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["unit"] == "points/s" and d["higher_is_better"]
    assert d["warmup"] >= 3                                   # the warm-up floor is enforced
    assert d["steps"] == 2 and d["value"] > 0
    assert d["config"]["workload"] == "tiny"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "points/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    # value = sampled points of one step / the mean step time
    pts = int(d["cpu_baseline"]["sample"].split("(")[1].split()[0])
    assert abs(d["value"] - pts / (d["ms_per_step"] / 1e3)) <= 1e-6 * d["value"]
