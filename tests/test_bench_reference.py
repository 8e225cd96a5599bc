"""bench.py's reference arm (the oracle on the host cores) runs on a machine
without a GPU and prints one JSON line with the contract's keys."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3",
                        "--warmup", "3", "--batch", "20000"], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    res = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "cpu_baseline", "e2e", "config"):
        assert k in res, k
    assert res["impl"] == "reference" and res["value"] > 0
    assert res["e2e"]["h2d_bytes_per_step"] == 0 and res["cpu_baseline"]["kind"] == "oracle"
