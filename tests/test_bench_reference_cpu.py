"""The reference arm of bench.py (the CPU oracle timed on the host cores)
runs without a GPU: one JSON line with the GPU arm's metric, unit and
config, on rank 0 only."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          env=e, capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_contract_line():
    r = run_bench("--impl", "reference", "--steps", "1", "--warmup", "0")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    j = json.loads(lines[0])
    sys.path.insert(0, ROOT)
    import bench
    assert j["impl"] == "reference"
    assert j["metric"] == bench.METRIC and j["unit"] == "tokens/s"
    assert j["higher_is_better"] is True and j["scaling"] == "weak"
    assert j["n_gpus"] == 1 and j["steps"] == 1 and j["warmup"] == 0
    assert j["value"] > 0 and j["ms_per_step"] > 0
    assert j["vs_baseline"] is None and j["data"] == "synthetic" and j["dtype"] == "bf16"
    assert j["config"]["R"] == 8 and j["config"]["T"] == 8192 and j["config"]["H"] == 7168
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == j["value"]
    assert cb["sample"]
    assert j["e2e"] == {"value": j["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert j["gpu_launches"] == 0


def test_reference_arm_other_ranks_exit_without_work():
    r = run_bench("--impl", "reference", "--steps", "1", "--warmup", "0",
                  env={"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{")]


def test_algorithmic_bytes_of_the_benchmarked_workload():
    # 8 partials + residual_in + residual_out (bf16) + NVFP4 codes + E4M3 block
    # scales of 8192 x 7168: 939,524,096 + 2 x 117,440,512 + 29,360,128 + 3,670,016
    sys.path.insert(0, ROOT)
    import bench
    assert bench.algorithmic_bytes(8, 8192, 7168) == 1_207_435_264
    assert bench.algorithmic_bytes(1, 1, 16) == 16 * 2 * 3 + 8 + 1
