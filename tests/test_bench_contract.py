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


def test_peak_choice_by_timing_window():
    import bench
    peaks = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    p, src = bench.choose_peak(peaks, "measured", 0.05)
    assert p == 1900.0 and "burst" in src
    p, src = bench.choose_peak(peaks, "measured", 4.0)
    assert p == 1700.0 and "sustained" in src


def test_reference_covers_whole_steps_where_affordable():
    import bench
    from matrix_aware_optimizers_gb300 import workloads
    assert bench.reference_items(workloads.workload(1)) == 4      # every worker
    assert bench.reference_items(workloads.workload(2)) == 48     # every matrix
    assert bench.reference_items(workloads.workload(3)) == 1      # one 4096^2 worker
    assert bench.reference_items(workloads.workload(4)) == 1
    assert 1 < bench.reference_items(workloads.workload(5)) < 385


def test_both_arms_describe_the_same_config():
    # the GPU arm and the oracle arm build the config from the workload and the flags only
    import bench
    from matrix_aware_optimizers_gb300 import workloads
    wl = workloads.workload(2)
    d = _run("--impl", "reference", "--config", "2", "--steps", "1", "--warmup", "1")
    assert d["config"] == json.loads(json.dumps(bench.config_block(wl, "bits", False, None, 1)))
    assert d["step_fraction"] == 1.0
    assert abs(d["value"] * d["ms_per_step"] / 1000.0 - 1.0) < 0.05


def test_per_config_entries_name_existing_parity_tests():
    """Every workload the default line measures under per_config names the GPU parity tests
    that check it, and those tests exist."""
    sys.path.insert(0, ROOT)
    import bench
    src = open(os.path.join(ROOT, "tests", "test_gpu_steps.py")).read()
    assert set(bench.PER_CONFIG) <= set(bench.PARITY_TESTS)
    for c, names in bench.PARITY_TESTS.items():
        for name in names.replace("tests/test_gpu_steps.py::", "").split(","):
            assert "def %s(" % name.strip() in src, (c, name)
