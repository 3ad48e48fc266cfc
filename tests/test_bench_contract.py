"""The benchmark's output contract, checked on the reference arm (the oracle on
the host's cores, so it runs without a GPU): one JSON line with the keys the
measurement contract names, the reference arm's marker and its zero-copy e2e
object, and consistent throughput arithmetic."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.strip().splitlines() if l.strip()]
    assert len(lines) == 1, lines
    return json.loads(lines[0])


def test_reference_arm_line():
    d = _run("--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "3")
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] >= 3
    assert d["unit"] == "tok/s" and d["higher_is_better"] is True and d["data"] == "synthetic"
    assert d["config"]["workload"] and d["config"]["shape"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
    # tokens per second and milliseconds per step agree (B = 1 slot)
    assert abs(d["value"] * d["ms_per_step"] / 1e3 - d["config"]["B"]) < 1e-6 * d["config"]["B"] + 1e-9
