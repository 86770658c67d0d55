"""Host-side logic of bench.py, without a GPU: the max-over-ranks aggregation under a real
two-rank gloo process group, the whole-job throughput, the clock-sample parser, the traffic
lines (accepted only for the library build that is running), the peak chosen by the timed
region's length, the secondary workloads' parser, the summary of a timed workload, and the
algorithmic byte counts."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, rank, world)
        # rank r measured a step of (r + 1) ms and an e2e time of (10 - r) ms
        got = bench.max_over_ranks([rank + 1.0, 10.0 - rank], dist)
        dist.barrier()
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results[0] == results[1] == [2.0, 10.0]


def test_max_over_ranks_without_a_group_is_identity():
    assert bench.max_over_ranks([1, 2.5]) == [1.0, 2.5]


def test_whole_job_throughput_counts_every_rank():
    w = synth.WORKLOADS["7b"]
    one = bench.whole_job_tflops(1, w.flops, 1.0)
    assert abs(one - w.flops / 1e-3 / 1e12) < 1e-9
    assert abs(bench.whole_job_tflops(8, w.flops, 1.0) - 8 * one) < 1e-6


def test_clock_sampler_parses_and_windows(tmp_path):
    cs = bench.ClockSampler(0)
    path = tmp_path / "clocks.csv"
    path.write_text(
        "2026/12/02 06:00:00.000, 1500, 2070, 900.0, 0x4, Not Active, Not Active, Not Active, Active\n"
        "2026/12/02 06:00:01.000, 1700, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active\n"
        "2026/12/02 06:00:02.000, 1900, 2070, 1350.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
        "garbage line\n")
    import datetime
    t = datetime.datetime(2026, 12, 2, 6, 0, 0).timestamp()

    class FakeProc:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    cs.proc, cs.path, cs.fh = FakeProc(), str(path), open(path, "a")
    cs.t0, cs.t1 = t + 0.5, t + 2.5  # the last two samples fall inside the timed window
    got = cs.stop()
    assert got["samples"] == 2 and got["sm_mhz"] == 1800.0 and got["sm_max_mhz"] == 2070.0
    assert got["reasons"] == ["sw_power_cap"] and got["window"] == "timed region"


def test_traffic_lines_need_the_running_build(tmp_path, monkeypatch):
    f = tmp_path / "traffic.txt"
    f.write_text("# DRAM bytes per launch\n"
                 "traffic gpt3-175b gemm2 5100000000 build 0123456789abcdef\n"
                 "traffic 7b gemm2 1310000000 build fedcba9876543210\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    v, why = bench.measured_traffic("gpt3-175b", "gemm2", "0123456789abcdef")
    assert v == 5.1e9 and "0123456789abcdef" in why
    v, why = bench.measured_traffic("7b", "gemm2", "0123456789abcdef")
    assert v is None and "another build" in why
    v, why = bench.measured_traffic("7b", "gemm1", "0123456789abcdef")
    assert v is None and "no capture" in why
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "absent.txt"))
    assert bench.measured_traffic("7b", "gemm2", "x")[0] is None


def test_committed_traffic_lines_are_well_formed():
    if not os.path.exists(bench.TRAFFIC_FILE):
        pytest.skip("no traffic summary committed")
    import re
    n = 0
    for ln in open(bench.TRAFFIC_FILE):
        if ln.startswith("traffic "):
            parts = ln.split()
            assert len(parts) == 6 and parts[4] == "build", ln
            assert parts[1] in synth.WORKLOADS or parts[1].startswith("custom-"), ln
            assert parts[2] in ("gemm1", "gemm2") and float(parts[3]) > 1e6, ln
            assert re.fullmatch(r"[0-9a-f]{16}", parts[5]), ln
            n += 1
    assert n >= 1


def test_peak_follows_the_timed_region():
    peaks = {"bf16_tflops": 1960.6, "bf16_tflops_sustained": 1734.7, "hbm_gbs": 6750.0}
    assert bench.peak_for(peaks, 0.12) == (1960.6, "burst")
    assert bench.peak_for(peaks, bench.BURST_LIMIT_S + 0.5) == (1734.7, "sustained")
    assert bench.peak_for({"bf16_tflops": 1900.0}, 5.0) == (1900.0, "sustained")


def test_secondary_spec():
    got = bench.parse_secondary("7b,gpt2-small,sweep-h4096:1/8/16")
    assert got == [("7b", (8,)), ("gpt2-small", (4,)), ("sweep-h4096", (1, 8, 16))]
    assert bench.parse_secondary("") == []
    with pytest.raises(ValueError):
        bench.parse_secondary("no-such-workload")
    with pytest.raises(ValueError):
        bench.parse_secondary("7b:3")  # 16384 / 3 is not a whole number of 64-column blocks


def test_summary_of_a_timed_workload():
    w = synth.WORKLOADS["gpt3-175b"]
    peaks = {"bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0, "hbm_gbs": 6750.0}
    res = {"ms_step": 5.0, "t_wall": 0.3, "kernel_ms": {"gemm1": 2.4, "gemm2": 2.6},
           "ln_ms": None}
    s = bench.summarize(w, "gelu", res, 1, peaks)
    assert s["value"] == pytest.approx(w.flops / 5e-3 / 1e12)
    assert s["peak_regime"] == "burst"
    assert s["pct_of_dense_bf16_peak"] == pytest.approx(100 * s["value"] / 2000.0)
    assert s["pct_of_dense_bf16_peak_sustained"] == pytest.approx(100 * s["value"] / 1600.0)
    r = s["roofline"]
    assert r["kernel"] == "gemm2" and r["peak"] == 2000.0
    assert r["achieved"] == pytest.approx(2 * w.M * w.H * w.F / 2.6e-3 / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / 2000.0)
    assert r["frac_sustained"] == pytest.approx(r["achieved"] / 1600.0)
    hb = s["hbm_gbs_algorithmic"]
    assert hb["step"] == pytest.approx(bench.block_bytes(w) / 5e-3 / 1e9)
    assert hb["step_with_y"] == pytest.approx((bench.block_bytes(w) + 4 * w.M * w.F) / 5e-3 / 1e9)
    res["t_wall"] = 3.0
    assert bench.summarize(w, "gelu", res, 1, peaks)["roofline"]["peak"] == 1600.0


def test_algorithmic_bytes():
    w = synth.WORKLOADS["7b"]
    g1 = bench.alg_bytes(w, "gemm1")
    assert g1 == 2 * w.M * w.H + 2 * w.H * w.F + 4 * w.F + 2 * w.M * w.F
    assert bench.alg_bytes(w, "gemm1", "swiglu") == g1 + 2 * w.H * w.F + 4 * w.F
    assert bench.alg_bytes(w, "gemm2", "block") == bench.alg_bytes(w, "gemm2") + 2 * w.M * w.H
    assert bench.step_flops(w, "swiglu") == 6 * w.M * w.H * w.F
    assert bench.step_flops(w, "gelu") == 4 * w.M * w.H * w.F
    # X in, Z out, W1, W2 and both biases once
    assert bench.block_bytes(w) == 4 * w.M * w.H + 4 * w.H * w.F + 4 * w.F + 4 * w.H


def test_clock_sampler_queries_the_process_gpu(monkeypatch):
    """nvidia-smi -i gets the device's UUID when torch has one, else the CUDA_VISIBLE_DEVICES
    entry of the CUDA ordinal (ordinals are renumbered by it, nvidia-smi indices are not),
    else the ordinal."""
    u = "3f2a9c1e-0b7d-4e55-9a21-6c0d8e4b7f10"
    assert bench.smi_gpu_id(0, uuid=u) == "GPU-" + u
    assert bench.smi_gpu_id(0, uuid="GPU-" + u) == "GPU-" + u
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "3,5")
    assert bench.smi_gpu_id(1, uuid="not-a-uuid") == "5"
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "GPU-" + u)
    assert bench.smi_gpu_id(0, uuid="") == "GPU-" + u
    monkeypatch.delenv("CUDA_VISIBLE_DEVICES")
    assert bench.smi_gpu_id(2, uuid="") == "2"
