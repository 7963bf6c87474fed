"""bench.py's reference arm (the fp64 oracle on the host cores) prints one JSON line with
the keys the benchmark contract names. CPU only: the reference arm never touches a GPU."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


def test_reference_arm_json_line():
    d = _run("--impl", "reference", "--config", "1", "--steps", "2", "--warmup", "1")
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True and d["unit"] == "steps/s"
    assert d["config"]["workload"] == "signmuon_64x128_f32_w4"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    e = d["e2e"]
    assert e["value"] == d["value"] and e["h2d_bytes_per_step"] == 0 == e["d2h_bytes_per_step"]


def test_reference_arm_variants_and_dion():
    d = _run("--impl", "reference", "--config", "1", "--steps", "1", "--warmup", "1",
             "--variant", "int8", "--post-polar")
    assert d["config"]["aggregation"].startswith("int8") and d["config"]["post_vote_polar"]
    d = _run("--impl", "reference", "--config", "6", "--steps", "1", "--warmup", "1")
    assert d["metric"].startswith("Dion") and d["value"] > 0
