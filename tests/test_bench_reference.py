"""The benchmark's reference arm on the CPU: `bench.py --impl reference` times the fp64 oracle
on the host cores and prints one JSON line with the GPU arm's metric, unit and direction, plus
the keys the line of a reference run carries (impl, cpu_baseline, e2e with no copies).

Run as the driver runs it, in a subprocess: on the default (GPT-3-175B-shaped) workload with a
small time budget, on the tiny workload, and as a second rank under a torchrun-style environment, which
must exit 0 without output (only rank 0 times the oracle)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def run_bench(*args, env_extra=None, timeout=240):
    env = dict(os.environ)
    env.update(env_extra or {})
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       env=env, capture_output=True, text=True, timeout=timeout)
    assert p.returncode == 0, p.stderr[-2000:]
    return p.stdout


@pytest.mark.parametrize("workload,extra", [
    ("gpt3-175b", ["--reference-budget-s", "3"]),   # the default workload, bounded sample
    ("tiny", ["--reference-budget-s", "2"]),
])
def test_reference_arm_line(workload, extra):
    out = run_bench("--impl", "reference", "--workload", workload, "--steps", "2", "--warmup",
                    "3", *extra)
    lines = [ln for ln in out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "TFLOP/s"
    assert line["higher_is_better"] is True and line["n_gpus"] == 1
    assert line["steps"] == 2 and line["warmup"] == 3
    assert line["value"] > 0 and line["ms_per_step"] > 0 and line["tokens_per_s"] > 0
    assert line["gpu_launches"] == 0
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert "token rows" in cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    cfg = line["config"]
    assert cfg["M"] == bench.synth.WORKLOADS[workload].M
    assert 1 <= cfg["rows_per_step"] <= cfg["M"]
    # the throughput is the sampled rows' FLOPs over the step time
    want = cfg["rows_per_step"] * cfg["flops_per_step"] // cfg["M"] / (line["ms_per_step"] * 1e-3)
    assert abs(line["value"] * 1e12 - want) <= 1e-6 * want


def test_reference_arm_other_ranks_print_nothing():
    out = run_bench("--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3",
                    env_extra={"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"})
    assert out.strip() == ""
