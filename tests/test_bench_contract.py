"""bench.py's reference arm (the oracle timed on the host cores) keeps the
JSON-line contract: one line with the metric, the timing keys, a
cpu_baseline describing the run and an e2e object without copies. Runs on
CPU with the small fp32 configuration."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_reference_arm_json_line():
    d = _run("--impl", "reference", "--preset", "tiny_t256_d512_e16_fp32", "--steps", "2", "--warmup", "1")
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference"
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == "tiny_t256_d512_e16_fp32"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_print_nothing():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", RANK="1", LOCAL_RANK="1", WORLD_SIZE="2",
               MASTER_ADDR="127.0.0.1", MASTER_PORT="29555")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--preset", "tiny_t256_d512_e16_fp32", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_clock_samples_are_taken_from_the_timed_region():
    """The clocks summary keeps the nvidia-smi samples stamped inside the
    timed region (all samples when none are) and reports throttle reasons."""
    import datetime
    sys.path.insert(0, ROOT)
    import bench
    lines = ["2026/12/03 10:00:00.100, 0, 1300, 2032, 900.5, 0x4, Not Active, Not Active, Not Active, Active",
             "2026/12/03 10:00:00.150, 0, 1350, 2032, 950.5, 0x4, Not Active, Not Active, Not Active, Active",
             "2026/12/03 10:00:01.150, 0, 1900, 2032, 150.5, 0x0, Not Active, Not Active, Not Active, Not Active",
             "garbled line"]
    t0, t1 = datetime.datetime(2026, 12, 3, 10, 0, 0), datetime.datetime(2026, 12, 3, 10, 0, 1)
    s = bench.ClockSampler.parse(lines, t0, t1)
    assert s["samples_in_timed_region"] == 2 and s["sm_mhz"] == 1325.0 and s["power_w_median"] == 925.5
    assert s["reasons"] == ["sw_power_cap"] and s["sm_max_mhz"] == 2032.0
    s = bench.ClockSampler.parse(lines)
    assert s["samples"] == 3 and s["samples_in_timed_region"] == 0 and s["sm_mhz"] == 1350.0
    assert bench.ClockSampler.parse(["garbled"]) is None
