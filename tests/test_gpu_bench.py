"""The benchmark's GPU arm end to end on the tiny workload: `bench.py` runs as the driver runs
it (a subprocess, one GPU) and prints one JSON line that carries every key of the contract --
the metric and its unit, the step timing, the roofline of the dominant kernel against the
measured peak, the end-to-end number through the host-buffer entry point with the bytes it
copies, the launch count, the clocks sampled during the timed region and the oracle's CPU
baseline."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

pytestmark = pytest.mark.gpu


def bench_line(*args):
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-3000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("variant", ["gelu", "swiglu"])
def test_bench_line_carries_the_contract(lib, variant):
    steps = 20
    line = bench_line("--workload", "tiny", "--variant", variant, "--steps", str(steps),
                      "--warmup", "3", "--cpu-budget-s", "1", "--secondary", "")
    w = bench.synth.WORKLOADS["tiny"]
    assert line["metric"] == bench.METRIC and line["unit"] == "TFLOP/s"
    assert line["n_gpus"] == 1 and line["steps"] == steps and line["warmup"] == 3
    assert line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["vs_baseline"] is None and line["dtype"] == "bf16"
    assert line["data"].startswith("synthetic")
    cfg = line["config"]
    assert cfg["M"] == w.M and cfg["H"] == w.H and cfg["F"] == w.F and cfg["k"] == w.k
    assert cfg["variant"] == variant and "workload" in cfg and "l2" in cfg
    # value = the step's FLOPs over its mean device time
    assert line["value"] > 0
    want = cfg["flops_per_step"] / (line["ms_per_step"] * 1e-3) / 1e12
    assert abs(line["value"] - want) <= 1e-6 * want
    roof = line["roofline"]
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s"
    assert roof["peak"] > 0 and roof["achieved"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) <= 1e-9
    # a 20-step tiny run is far under a second of work: compared with the burst peak
    assert line["peak_regime"] == roof["peak_regime"] == "burst"
    assert line["timed_region_s"] < bench.BURST_LIMIT_S
    assert roof["frac_burst"] == roof["frac"] and roof["frac_sustained"] >= roof["frac"]
    assert "traffic" in roof and "traffic_source" in roof
    assert len(line["build_id"]) == 16
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == "TFLOP/s"
    assert e2e["h2d_bytes_per_step"] == w.M * w.H * 2 == e2e["d2h_bytes_per_step"]
    assert "tpmlp_host_wait" in e2e["api"] and e2e["steps"] >= 3
    sync = e2e["synchronous_calls"]
    assert sync["value"] > 0 and abs(sync["value"] * sync["ms_per_step"] -
                                     e2e["value"] * e2e["ms_per_step"]) <= 1e-6 * e2e["value"] * e2e["ms_per_step"]
    assert line["gpu_launches"] == 2 * steps  # two GEMM launches per forward
    clk = line["clocks"]
    assert clk is not None and clk["sm_mhz"] > 0 and clk["sm_max_mhz"] >= clk["sm_mhz"]
    assert isinstance(clk["reasons"], list)
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0
    assert "token rows" in cb["sample"]


def test_bench_secondary_workloads(lib):
    """The secondary workloads are timed in the same process and reported with their own
    throughput, kernel times, roofline and HBM figures; a sweep reports every shard count."""
    line = bench_line("--workload", "tiny", "--steps", "5", "--warmup", "3", "--no-cpu-baseline",
                      "--secondary", "gpt2-small,tiny:1/2")
    sec = line["secondary"]
    assert sorted(sec) == ["gpt2-small", "tiny-k1", "tiny-k2"]
    for label, s in sec.items():
        cfg = s["config"]
        want = cfg["flops_per_step"] / (s["ms_per_step"] * 1e-3) / 1e12
        assert abs(s["value"] - want) <= 1e-6 * want, label
        assert s["gpu_launches"] == 2 * 5, label
        assert set(s["kernel_ms"]) == {"gemm1", "gemm2"}
        assert s["roofline"]["kernel"] in ("gemm1", "gemm2")
        assert s["hbm_gbs_algorithmic"]["step"] > 0
        assert s["peak_regime"] == "burst"
    assert sec["tiny-k1"]["config"]["k"] == 1 and sec["tiny-k2"]["config"]["k"] == 2
    assert sec["gpt2-small"]["config"]["M"] == 8192
