"""The JSON line of the bench's reference arm (the fp64 oracle timed on the
host cores) on the small workload: one line, the keys the driver reads, and
values that describe this run."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_complete_json_line():
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "tiny_T256_E8_k2_h64_I32", "--steps", "2", "--warmup", "3"],
                         env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    r = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in r, key
    assert r["impl"] == "reference" and r["n_gpus"] == 1 and r["steps"] == 2 and r["warmup"] == 3
    assert r["higher_is_better"] is True and r["value"] > 0
    assert r["config"]["workload"] == "tiny_T256_E8_k2_h64_I32"
    assert r["cpu_baseline"]["kind"] == "oracle" and r["cpu_baseline"]["cores"] >= 1
    assert r["cpu_baseline"]["value"] == r["value"]
    assert r["e2e"]["value"] == r["value"] and r["e2e"]["unit"] == r["unit"]
    assert r["e2e"]["h2d_bytes_per_step"] == 0 and r["e2e"]["d2h_bytes_per_step"] == 0
