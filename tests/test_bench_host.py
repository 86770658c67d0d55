"""Host-side logic of bench.py, without a GPU: the max-over-ranks aggregation under a real
two-rank gloo process group, the whole-job throughput, the clock-sample parser, the traffic
lines read from profiles/, and the algorithmic byte counts."""
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


def test_traffic_lines_are_read_from_profiles():
    v = bench.measured_traffic("7b", "gemm1")
    assert v is None or v > 1e8  # a DRAM byte count per launch when a capture is committed
    assert bench.measured_traffic("no-such-workload", "gemm1") is None


def test_algorithmic_bytes():
    w = synth.WORKLOADS["7b"]
    g1 = bench.alg_bytes(w, "gemm1")
    assert g1 == 2 * w.M * w.H + 2 * w.H * w.F + 4 * w.F + 2 * w.M * w.F
    assert bench.alg_bytes(w, "gemm1", "swiglu") == g1 + 2 * w.H * w.F + 4 * w.F
    assert bench.alg_bytes(w, "gemm2", "block") == bench.alg_bytes(w, "gemm2") + 2 * w.M * w.H
    assert bench.step_flops(w, "swiglu") == 6 * w.M * w.H * w.F
    assert bench.step_flops(w, "gelu") == 4 * w.M * w.H * w.F


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
