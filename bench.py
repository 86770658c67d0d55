"""Benchmark of the tensor-parallel MLP block forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload gpt3-175b]
                    [--secondary 7b,gpt2-small,sweep-h4096:1/8/16] [--impl reference]

A step is one forward pass of the whole block -- the column-parallel GEMM with its fused
bias + GeLU, then the row-parallel GEMM whose accumulator sums all k shards and adds b2 --
over one batch of seeded synthetic input already resident in HBM. L2 is flushed (a
256 MiB write, then a read of it, so no dirty line is left) between timed steps, outside
the timed events. The headline workload is the GPT-3-175B-shaped block (H = 12288, the
largest that the pages name). The printed JSON line carries throughput (TFLOP/s of the two
contractions, tokens/s) and its share of the dense bf16 peak of the timed region's regime
(burst under a second of continuous work, else sustained; both are reported), the roofline
of the dominant kernel, an end-to-end figure through the host-buffer entry point, SM clocks
sampled during the timed region, the fp64 CPU oracle timed on a bounded sample of the same
workload on this host's cores, and, under "secondary", the same measurements of the other
workloads (the 7B shape, GPT-2-small with its HBM GB/s, the shard-count sweep).

With N > 1 (torchrun), every rank runs an independent replica on its own GPU (the block
needs no exchange between replicas); ranks meet only at the timing barriers.

``--impl reference`` times the fp64 CPU oracle as the reference arm on the same workload
(rank 0 only; each step a bounded sample of token rows).
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "TP-MLP forward TFLOP/s and tokens/s on 1 GB300; % of dense BF16 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def l2_flush(buf):
    """Evict L2 between timed steps: write a buffer larger than L2, then read it back, so the
    next step starts on a cold L2 that holds no dirty lines (their write-back would otherwise
    land inside the next timed kernel). Both run outside the timed events."""
    buf.zero_()
    buf.view(-1).view(dtype=__import__("torch").int64).sum()


def step_flops(w: synth.Workload, variant: str) -> int:
    """FLOPs of one forward pass: 2*M*H*F per contraction (the gated block's first GEMM
    computes the gate and the up projection: twice that). LayerNorm and the residual add
    are O(M*H) and not counted."""
    return 6 * w.M * w.H * w.F if variant == "swiglu" else w.flops


def kernel_flops(w: synth.Workload, variant: str, kernel: str) -> int:
    base = 2 * w.M * w.H * w.F
    return 2 * base if (variant == "swiglu" and kernel == "gemm1") else base


def workload_config(w: synth.Workload, extra=None, variant: str = "gelu") -> dict:
    if variant == "gelu":
        desc = (f"{w.name} TP-MLP: X [B={w.B},S={w.S},H={w.H}] bf16, W1 [{w.H},{w.F}], "
                f"W2 [{w.F},{w.H}], erf GeLU, k={w.k} shards, seeded synthetic")
    elif variant == "block":
        desc = (f"{w.name} TP-MLP layer Z = X + MLP(LayerNorm(X)): X [B={w.B},S={w.S},H={w.H}] "
                f"bf16, W1 [{w.H},{w.F}], W2 [{w.F},{w.H}], erf GeLU, k={w.k} shards, seeded "
                f"synthetic")
    else:
        desc = (f"{w.name} gated TP-MLP: X [B={w.B},S={w.S},H={w.H}] bf16, Wg and Wu "
                f"[{w.H},{w.F}], W2 [{w.F},{w.H}], SwiGLU, k={w.k} shards, seeded synthetic")
    cfg = {
        "workload": desc, "variant": variant,
        "B": w.B, "S": w.S, "M": w.M, "H": w.H, "F": w.F, "k": w.k, "seed": w.seed,
        "flops_per_step": step_flops(w, variant),
        "l2": "flushed between timed steps (256 MiB write then read, outside the timed events)",
    }
    if extra:
        cfg.update(extra)
    return cfg


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def max_over_ranks(values, pg=None, device="cpu"):
    """Element-wise maximum of a list of floats over all ranks (identity without a group)."""
    if pg is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def whole_job_tflops(world: int, flops_per_rank_step: int, ms_per_step: float) -> float:
    """Throughput of all ranks together: every rank did flops_per_rank_step in the slowest
    rank's step time."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


# ------------------------------------------------------------------ clocks
_UUID_RE = re.compile(r"^GPU-[0-9a-fA-F]{8}(-[0-9a-fA-F]{4}){3}-[0-9a-fA-F]{12}$")


def smi_gpu_id(dev_index: int, uuid=None) -> str:
    """The id `nvidia-smi -i` takes for CUDA device `dev_index`. CUDA ordinals are renumbered
    under CUDA_VISIBLE_DEVICES and nvidia-smi's indices are not, so use the device's UUID
    (`uuid`: torch's for the device, looked up when not given), else the matching entry of
    CUDA_VISIBLE_DEVICES, else the ordinal itself."""
    if uuid is None:
        try:
            import torch
            uuid = torch.cuda.get_device_properties(dev_index).uuid
        except Exception:
            uuid = None
    if uuid is not None:
        u = str(uuid)
        u = u if u.startswith("GPU-") else "GPU-" + u
        if _UUID_RE.match(u):
            return u
    parts = [p.strip() for p in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if p.strip()]
    if 0 <= dev_index < len(parts):
        return parts[dev_index]
    return str(dev_index)


class ClockSampler:
    """nvidia-smi samples every 50 ms; stop() keeps the samples taken inside the timed window
    (mark_start / mark_stop) when there are any, else all of them (and says so)."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: str):
        self.gpu = gpu  # an id nvidia-smi -i accepts (smi_gpu_id)
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_stop(self):
        self.t1 = time.time()

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception as e:  # no nvidia-smi: record nothing
            log("clock sampling unavailable:", e)
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        import datetime
        rows = []
        with open(self.path) as fh:
            for ln in fh:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        inside = [r for r in rows if self.t0 is not None and self.t1 is not None
                  and self.t0 <= r[0] <= self.t1]
        use = inside or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        mx = max(r[2] for r in use)
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": mx,
                "reasons": reasons, "samples": len(use),
                "window": "timed region" if inside else "whole run (no sample fell inside the "
                                                         "timed region)"}


# ------------------------------------------------------------------ oracle (CPU) timing
def ln_params(H: int):
    return (synth.normal_bf16(5, 40, (H,), 0.5, mean=1.0), synth.normal_bf16(5, 41, (H,), 0.1))


def run_oracle(w: synth.Workload, d: dict, rows, variant: str):
    import oracle
    if variant == "gelu":
        return oracle.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], w.k, rows=rows)
    if variant == "block":
        g, b = ln_params(w.H)
        return oracle.block(d["X"], g, b, 1e-5, d["W1"], d["b1"], d["W2"], d["b2"], w.k,
                            rows=rows)
    return oracle.tpmlp_swiglu(d["X"], d["Wg"], d["bg"], d["Wu"], d["bu"], d["W2"], d["b2"], w.k,
                               rows=rows)


def oracle_sample(w: synth.Workload, d: dict, budget_s: float, max_rows: int,
                  variant: str = "gelu"):
    """Time the fp64 oracle on a bounded, seeded sample of token rows of the workload."""
    import oracle
    cal_rows = synth.sample_rows(w.M, min(max(oracle.threads(), 4), max_rows))
    t0 = time.perf_counter()
    run_oracle(w, d, cal_rows, variant)
    t_cal = time.perf_counter() - t0
    per_row = t_cal / len(cal_rows)
    R = int(max(len(cal_rows), min(max_rows, budget_s / max(per_row, 1e-9))))
    rows = synth.sample_rows(w.M, R)
    t0 = time.perf_counter()
    run_oracle(w, d, rows, variant)
    dt = time.perf_counter() - t0
    flops = len(rows) * step_flops(w, variant) // w.M
    return {"rows": len(rows), "seconds": dt, "tflops": flops / dt / 1e12,
            "tokens_per_s": len(rows) / dt, "cores": oracle.threads()}


# ------------------------------------------------------------------ reference arm
def run_reference(args, w: synth.Workload):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    import oracle
    v = args.variant
    d = synth.make_swiglu_inputs(w.H, w.F, w.M, w.seed) if v == "swiglu" else synth.workload_inputs(w)
    steps, warm = args.steps, args.warmup
    budget = args.reference_budget_s
    # rows per step so that the whole run stays within the budget
    cal_rows = synth.sample_rows(w.M, max(oracle.threads(), 4))
    t0 = time.perf_counter()
    run_oracle(w, d, cal_rows, v)
    per_row = (time.perf_counter() - t0) / len(cal_rows)
    R = int(max(1, min(w.M, budget / (steps + warm) / max(per_row, 1e-9))))
    rows = synth.sample_rows(w.M, R)
    for _ in range(warm):
        run_oracle(w, d, rows, v)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        run_oracle(w, d, rows, v)
        times.append(time.perf_counter() - t0)
    t = statistics.mean(times)
    flops = len(rows) * step_flops(w, v) // w.M
    value = flops / t / 1e12
    sample = (f"{len(rows)} of {w.M} token rows per step (seeded spread incl. first/last), full "
              f"weights, all {w.H} outputs; fp64 oracle, OpenMP over rows")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": steps, "warmup": warm, "ms_per_step": t * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "tokens_per_s": len(rows) / t,
        "config": workload_config(w, {"parallelism": "host cores (oracle)",
                                      "rows_per_step": len(rows)}, variant=v),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm
BURST_LIMIT_S = 1.0  # timed regions shorter than this run before the power cap bites


def peak_for(peaks: dict, timed_s: float):
    """The dense bf16 peak a timed region of `timed_s` seconds is compared with: the burst
    figure (cuBLAS best of 10) below BURST_LIMIT_S of continuous work, else the sustained one
    (a seconds-long cuBLAS loop under the power cap). Returns (peak, regime)."""
    burst = peaks["bf16_tflops"]
    sust = peaks.get("bf16_tflops_sustained", burst)
    if timed_s < BURST_LIMIT_S:
        return burst, "burst"
    return sust, "sustained"


def block_bytes(w: synth.Workload, variant: str = "gelu") -> int:
    """Bytes the block must move at least: X in, Z out, the weights and biases once (the
    intermediate Y stays out of this count)."""
    parts = 2 if variant == "swiglu" else 1
    return 2 * 2 * w.M * w.H + parts * (2 * w.H * w.F + 4 * w.F) + 2 * w.F * w.H + 4 * w.H


def to_device_bf16(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def time_block(args, w: synth.Workload, variant: str, dev, flush, barrier, d=None,
               headline: bool = False, pg=None, local_rank: int = 0):
    """Time `args.steps` forward passes of one block workload (after `args.warmup` untimed
    ones), each on an L2 flushed outside the timed events, then the same number of passes with
    an event between the kernels to attribute time to each. With `headline`, also sample the
    SM clocks over the timed region and time the host-buffer entry point end to end.
    Returns the measurements and the inputs."""
    import torch
    import tensor_transformer_mlp_tmem_gb300 as tp

    if d is None:
        d = (synth.make_swiglu_inputs(w.H, w.F, w.M, w.seed) if variant == "swiglu"
             else synth.workload_inputs(w))
    X = to_device_bf16(d["X"], dev).view(w.B, w.S, w.H)
    Z = torch.empty((w.B, w.S, w.H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    mlp = tp.TPMLP(w.H, w.F, w.k, swiglu=(variant == "swiglu"))
    if variant == "swiglu":
        mlp.pack_swiglu(*(to_device_bf16(d[n], dev) for n in ("Wg", "bg", "Wu", "bu", "W2", "b2")))
    else:
        mlp.pack(*(to_device_bf16(d[n], dev) for n in ("W1", "b1", "W2", "b2")))
    if variant == "block":
        g, b = ln_params(w.H)
        mlp.set_layernorm(to_device_bf16(g, dev), to_device_bf16(b, dev), 1e-5)
    mlp.reserve(w.M)
    torch.cuda.synchronize(dev)  # the raw weights are released: only the packed copies stay

    def step(ev=None):
        # one pass of the whole block through the entry point a user calls: tpmlp_forward
        # (GEMM1 (+b1, GeLU) then GEMM2 (sum over shards, +b2), launched back to back), or
        # tpmlp_block_forward for the "block" variant (LayerNorm, GEMM1, GEMM2 + residual)
        if ev is not None:
            ev[0].record(stream)
        if variant == "block":
            tp.tpmlp_block_forward(mlp.ctx, X, w.B, w.S, Z, stream)
        else:
            tp.tpmlp_forward(mlp.ctx, X, w.B, w.S, Z, stream)
        if ev is not None:
            ev[1].record(stream)

    def staged_step(ev):
        # the same launches, with the library recording an event between them to attribute
        # time to each kernel (the events cost the launches' overlap, so their sum is a little
        # above a step of the timed region)
        ev[0].record(stream)
        if variant == "block":
            tp.tpmlp_block_forward_marked(mlp.ctx, X, w.B, w.S, Z, ev[3], ev[1], stream)
        else:
            tp.tpmlp_forward_marked(mlp.ctx, X, w.B, w.S, Z, ev[1], stream)
        ev[2].record(stream)

    for _ in range(args.warmup):
        l2_flush(flush)
        step()
    for _ in range(args.warmup):
        l2_flush(flush)
        staged_step([torch.cuda.Event(enable_timing=True) for _ in range(4)])
    torch.cuda.synchronize(dev)
    rc, detail = mlp.status()
    if rc != tp.TPMLP_OK:
        raise RuntimeError(f"{w.name}: device status after warm-up: {detail:#x}")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    clocks = None
    if headline:
        clocks = ClockSampler(smi_gpu_id(local_rank))
        clocks.start()
        time.sleep(0.3)
    launches0 = mlp.launches
    barrier()
    torch.cuda.synchronize(dev)
    if clocks:
        clocks.mark_start()
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        l2_flush(flush)
        step(evs[i])
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall0
    if clocks:
        clocks.mark_stop()
    barrier()
    launches = mlp.launches - launches0
    clk = clocks.stop() if clocks else None
    rc, detail = mlp.status()
    if rc != tp.TPMLP_OK:
        raise RuntimeError(f"{w.name}: device status after timed steps: {detail:#x}")
    st = [e[0].elapsed_time(e[1]) for e in evs]

    # per-kernel attribution: the same number of steps, right after the timed region
    aevs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for i in range(args.steps):
        l2_flush(flush)
        staged_step(aevs[i])
    torch.cuda.synchronize(dev)
    if variant == "block":
        ln = [e[0].elapsed_time(e[3]) for e in aevs]
        g1 = [e[3].elapsed_time(e[1]) for e in aevs]
    else:
        ln = []
        g1 = [e[0].elapsed_time(e[1]) for e in aevs]
    g2 = [e[1].elapsed_time(e[2]) for e in aevs]
    ms_step = statistics.mean(st)
    ms_step, t_wall = max_over_ranks([ms_step, t_wall], pg, dev)
    res = {"ms_step": ms_step, "t_wall": t_wall, "launches": launches, "clocks": clk,
           "kernel_ms": {"gemm1": statistics.mean(g1), "gemm2": statistics.mean(g2)},
           "ln_ms": statistics.mean(ln) if ln else None}

    if headline:
        # end to end through the host-buffer entry point (pinned host memory)
        Xh = torch.from_numpy(np.ascontiguousarray(d["X"]).view(np.int16)).view(
            torch.bfloat16).pin_memory()
        Zh = torch.empty((w.M, w.H), dtype=torch.bfloat16).pin_memory()

        # a second output buffer, so that consecutive queued steps write different memory
        Zh2 = torch.empty((w.M, w.H), dtype=torch.bfloat16).pin_memory()

        def e2e_step():
            if variant == "block":
                tp.tpmlp_block_forward_host(mlp.ctx, Xh, w.B, w.S, Zh, stream)
            else:
                tp.tpmlp_forward_host(mlp.ctx, Xh, w.B, w.S, Zh, stream)

        def e2e_step_async(i):
            z = Zh if i % 2 == 0 else Zh2
            if variant == "block":
                tp.tpmlp_block_forward_host_async(mlp.ctx, Xh, w.B, w.S, z, stream)
            else:
                tp.tpmlp_forward_host_async(mlp.ctx, Xh, w.B, w.S, z, stream)

        e2e_steps = max(3, min(args.steps, 50))
        # (1) a stream of queued calls, one wait at the end: each step's input copy runs during
        # the previous step's kernels and its output copy during the next one's
        for i in range(max(1, args.warmup)):
            e2e_step_async(i)
        tp.tpmlp_host_wait(mlp.ctx)
        barrier()
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            e2e_step_async(i)
        tp.tpmlp_host_wait(mlp.ctx)
        e2e_s = (time.perf_counter() - t0) / e2e_steps
        # (2) one synchronous call per step (each returns with its Z in host memory)
        for _ in range(max(1, args.warmup)):
            e2e_step()
        barrier()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        e2e_sync_s = (time.perf_counter() - t0) / e2e_steps
        e2e_s, e2e_sync_s = max_over_ranks([e2e_s, e2e_sync_s], pg, dev)
        rc, detail = mlp.status()
        if rc != tp.TPMLP_OK:
            raise RuntimeError(f"{w.name}: device status after e2e steps: {detail:#x}")
        res["e2e_s"] = e2e_s
        res["e2e_sync_s"] = e2e_sync_s
        res["e2e_steps"] = e2e_steps
    mlp.close()
    del X, Z
    return res, d


def summarize(w: synth.Workload, variant: str, res: dict, world: int, peaks: dict):
    """Throughput, % of peak (the peak of the timed region's regime, and both), per-kernel
    times and the dominant kernel's roofline of one timed workload."""
    flops_step = step_flops(w, variant)
    value = whole_job_tflops(world, flops_step, res["ms_step"])
    peak, regime = peak_for(peaks, res["t_wall"])
    burst = peaks["bf16_tflops"]
    sust = peaks.get("bf16_tflops_sustained", burst)
    kern = res["kernel_ms"]
    kflops = {kk: kernel_flops(w, variant, kk) for kk in kern}
    dom = max(kern, key=lambda kk: kern[kk])
    achieved = kflops[dom] / (kern[dom] * 1e-3) / 1e12
    ln_ms = res["ln_ms"]
    out = {
        "value": value, "unit": "TFLOP/s", "ms_per_step": res["ms_step"],
        "tokens_per_s": world * w.M / (res["ms_step"] * 1e-3),
        "timed_region_s": res["t_wall"], "peak_regime": regime,
        "pct_of_dense_bf16_peak": 100.0 * (value / world) / peak,
        "pct_of_dense_bf16_peak_burst": 100.0 * (value / world) / burst,
        "pct_of_dense_bf16_peak_sustained": 100.0 * (value / world) / sust,
        "kernel_ms": dict(kern, **({"layernorm": ln_ms} if ln_ms else {})),
        "hbm_gbs_algorithmic": {  # algorithmic bytes of each launch / its mean event time
            "gemm1": alg_bytes(w, "gemm1", variant) / (kern["gemm1"] * 1e-3) / 1e9,
            "gemm2": alg_bytes(w, "gemm2", variant) / (kern["gemm2"] * 1e-3) / 1e9,
            **({"layernorm": (4 * w.M * w.H + 8 * w.H) / (ln_ms * 1e-3) / 1e9} if ln_ms else {}),
            # the block's X, Z, weights and biases once per step (Y excluded), and with the
            # round trip of Y through HBM that two launches add
            "step": block_bytes(w, variant) / (res["ms_step"] * 1e-3) / 1e9,
            "step_with_y": (block_bytes(w, variant) + 4 * w.M * w.F) / (res["ms_step"] * 1e-3) / 1e9,
            "peak_hbm_gbs": peaks["hbm_gbs"]},
        "roofline": {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak,
                     "frac_burst": achieved / burst, "frac_sustained": achieved / sust,
                     "peak_regime": regime},
    }
    return out


def run_gpu(args, w: synth.Workload):
    import torch
    import tensor_transformer_mlp_tmem_gb300 as tp

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    def barrier():
        if pg is not None:
            pg.barrier()

    variant = args.variant
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    res, d = time_block(args, w, variant, dev, flush, barrier, headline=True, pg=pg,
                        local_rank=local_rank)
    peaks, peak_src = load_peaks()
    summ = summarize(w, variant, res, world, peaks)
    flops_step = step_flops(w, variant)
    dom = summ["roofline"]["kernel"]
    traffic, traffic_src = measured_traffic(w.name if variant == "gelu" else f"{w.name}-{variant}",
                                            dom, tp.tpmlp_build_id())
    regime = summ["peak_regime"]
    roofline = dict(summ["roofline"])
    roofline.update({
        "peak_source": (f"{peak_src} bf16_tflops ({'cuBLAS bf16 best of 10' if regime == 'burst' else 'cuBLAS bf16 loop under the power cap'}): "
                        f"the timed region ran {res['t_wall']:.3f} s, "
                        f"{'under' if regime == 'burst' else 'over'} {BURST_LIMIT_S:g} s of "
                        f"continuous work"),
        "traffic": traffic, "traffic_source": traffic_src})

    line = {
        "metric": METRIC, "value": summ["value"], "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": summ["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) X, N(0,1/fan_in) weights, N(0,0.02^2) biases)",
        "tokens_per_s": summ["tokens_per_s"],
        "pct_of_dense_bf16_peak": summ["pct_of_dense_bf16_peak"],
        "pct_of_dense_bf16_peak_burst": summ["pct_of_dense_bf16_peak_burst"],
        "pct_of_dense_bf16_peak_sustained": summ["pct_of_dense_bf16_peak_sustained"],
        "peak_regime": regime, "timed_region_s": res["t_wall"],
        "wall_ms_per_step_incl_l2_flush": res["t_wall"] * 1e3 / args.steps,
        "kernel_ms": summ["kernel_ms"],
        "kernel_ms_source": "CUDA events the library records between the launches "
                            "(tpmlp_forward_marked), over a pass of the same number of steps "
                            "right after the timed region (same L2 flush)",
        "hbm_gbs_algorithmic": summ["hbm_gbs_algorithmic"],
        "config": workload_config(w, {"parallelism": "replicas" if world > 1 else "single GPU",
                                      "output": "bf16"}, variant=variant),
        "roofline": roofline,
        "e2e": {"value": world * flops_step / res["e2e_s"] / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": w.M * w.H * 2, "d2h_bytes_per_step": w.M * w.H * 2,
                "ms_per_step": res["e2e_s"] * 1e3, "steps": res["e2e_steps"],
                "api": (("tpmlp_block_forward_host_async" if variant == "block"
                         else "tpmlp_forward_host_async")
                        + " + tpmlp_host_wait: the steps queued back to back from pinned host X "
                          "into two pinned host Z buffers, one wait at the end; each step's "
                          "input copy overlaps the previous step's kernels and its output copy "
                          "the next one's; host wall clock from the first call to the wait"),
                "synchronous_calls": {
                    "value": world * flops_step / res["e2e_sync_s"] / 1e12,
                    "ms_per_step": res["e2e_sync_s"] * 1e3,
                    "api": (("tpmlp_block_forward_host" if variant == "block"
                             else "tpmlp_forward_host")
                            + " (one call per step, returning with Z in host memory; planned "
                              "row chunks, copies overlapped with the kernels of the same "
                              "call)")}},
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
        "build_id": tp.tpmlp_build_id(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = oracle_sample(w, d, args.cpu_budget_s, args.cpu_max_rows, variant)
        line["cpu_baseline"] = {
            "value": cb["tflops"], "unit": "TFLOP/s", "cores": cb["cores"], "kind": "oracle",
            "sample": f"{cb['rows']} of {w.M} token rows (seeded spread incl. first/last), full "
                      f"weights, all {w.H} outputs; {cb['seconds']:.1f} s; fp64 plain loops, "
                      f"OpenMP over rows",
            "tokens_per_s": cb["tokens_per_s"]}
    del d

    # the other workloads of the same block, timed the same way in this process
    if variant == "gelu" and args.secondary:
        sec = {}
        for name, ks in parse_secondary(args.secondary):
            base = synth.WORKLOADS[name]
            dd = synth.workload_inputs(base)  # identical inputs for every k of a sweep
            for k in ks:
                ws = synth.Workload(base.name, base.B, base.S, base.H, base.F, k, base.seed)
                r, _ = time_block(args, ws, variant, dev, flush, barrier, d=dd, pg=pg)
                sm = summarize(ws, variant, r, world, peaks)
                sm["config"] = {"workload": f"{ws.name}: X [B={ws.B},S={ws.S},H={ws.H}], "
                                            f"W1 [{ws.H},{ws.F}], W2 [{ws.F},{ws.H}], k={ws.k}",
                                "M": ws.M, "H": ws.H, "F": ws.F, "k": ws.k,
                                "flops_per_step": step_flops(ws, variant)}
                sm["gpu_launches"] = r["launches"]
                label = ws.name if len(ks) == 1 and k == base.k else f"{ws.name}-k{k}"
                sec[label] = sm
            del dd
        line["secondary"] = sec
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.barrier()
        pg.destroy_process_group()
    return 0


def parse_secondary(spec: str):
    """"7b,gpt2-small,sweep-h4096:1/8/16" -> [("7b", (8,)), ("gpt2-small", (4,)),
    ("sweep-h4096", (1, 8, 16))]: each workload at its own shard count unless ":k1/k2/..."
    names the shard counts to time."""
    out = []
    for item in [p.strip() for p in spec.split(",") if p.strip()]:
        name, _, ks = item.partition(":")
        if name not in synth.WORKLOADS:
            raise ValueError(f"unknown workload {name!r} in --secondary")
        w = synth.WORKLOADS[name]
        kk = tuple(int(x) for x in ks.split("/")) if ks else (w.k,)
        for k in kk:
            if k <= 0 or w.F % k or (w.F // k) % 64:
                raise ValueError(f"shard count {k} does not divide {name}'s F={w.F} into "
                                 f"multiples of 64")
        out.append((name, kk))
    return out


def alg_bytes(w: synth.Workload, kernel: str, variant: str = "gelu") -> int:
    """Bytes a launch must move at least: its operands once and its output once
    (GEMM1: X, W1 (gated: Wg and Wu), biases, Y; GEMM2: Y, W2, b2, Z; bf16 tensors, fp32
    biases)."""
    if kernel == "gemm1":
        parts = 2 if variant == "swiglu" else 1
        return 2 * w.M * w.H + parts * (2 * w.H * w.F + 4 * w.F) + 2 * w.M * w.F
    residual = 2 * w.M * w.H if variant == "block" else 0
    return 2 * w.M * w.F + 2 * w.F * w.H + 4 * w.H + 2 * w.M * w.H + residual


def run_gpu_linear(args, w: synth.Workload):
    """The tensor-parallel attention projections on the workload's shape: "outproj" is the
    row-parallel output projection (K = N = H, heads split into k groups, the sum over
    shards in the accumulator), "qkv" the column-parallel Q/K/V projection (K = H, N = 3H)."""
    import torch
    import tensor_transformer_mlp_tmem_gb300 as tp

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    kind = "row" if args.variant == "outproj" else "column"
    K, N, M = w.H, (w.H if kind == "row" else 3 * w.H), w.M
    X = synth.normal_bf16(w.seed, 50, (M, K), 1.0)
    W = synth.normal_bf16(w.seed, 51, (K, N), 1.0 / np.sqrt(K))
    b = synth.normal_bf16(w.seed, 52, (N,), 0.02)

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    Xd, out = to_dev(X), torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    lin = tp.Linear(kind, K, N, w.k)
    lin.pack(to_dev(W), to_dev(b))
    for _ in range(args.warmup):
        l2_flush(flush)
        tp.tpmlp_linear_forward(lin.ctx, Xd, M, out, stream)
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    clocks = ClockSampler(smi_gpu_id(local_rank))
    clocks.start()
    time.sleep(0.3)
    n0 = tp.tpmlp_launch_count(lin.ctx)
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize(dev)
    clocks.mark_start()
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        l2_flush(flush)
        evs[i][0].record(stream)
        tp.tpmlp_linear_forward(lin.ctx, Xd, M, out, stream)
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall0
    clocks.mark_stop()
    if pg is not None:
        pg.barrier()
    launches = tp.tpmlp_launch_count(lin.ctx) - n0
    clk = clocks.stop()
    rc, detail = lin.status()
    if rc != tp.TPMLP_OK:
        raise RuntimeError(f"device status {detail:#x}")
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    (ms,) = max_over_ranks([ms], pg, dev)
    flops = 2 * M * K * N
    peaks, peak_src = load_peaks()
    peak, regime = peak_for(peaks, t_wall)
    value = whole_job_tflops(world, flops, ms)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) X, N(0,1/K) W)",
        "peak_regime": regime, "timed_region_s": t_wall,
        "tokens_per_s": world * M / (ms * 1e-3),
        "config": {"workload": f"{w.name}-shaped attention {'output' if kind == 'row' else 'Q/K/V'} "
                               f"projection: X [{M},{K}] bf16, W [{K},{N}], {kind}-parallel, "
                               f"k={w.k} head groups, seeded synthetic",
                   "variant": args.variant, "M": M, "K": K, "N": N, "k": w.k,
                   "flops_per_step": flops,
                   "l2": "flushed between timed steps (256 MiB write then read, outside the timed events)"},
        "roofline": {"bound": "tensor", "kernel": f"{kind}-parallel linear", "achieved": value / world,
                     "peak": peak, "unit": "TFLOP/s", "frac": value / world / peak,
                     "peak_source": f"{peak_src} bf16_tflops ({regime})", "traffic": None},
        "gpu_launches": launches, "clocks": clk,
    }
    lin.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.barrier()
        pg.destroy_process_group()
    return 0


def run_gpu_train(args, w: synth.Workload):
    """One training step of the block: tpmlp_forward_train (keeps Y and the pre-activation)
    then tpmlp_backward (dA, dX summed over shards in the accumulator, dW1, dW2, db1, db2).
    FLOPs: forward 4 M H F, backward 8 M H F (four GEMMs of 2 M H F each).
    Gated block (--variant train-swiglu): tpmlp_forward_train (keeps Y, G and U) then
    tpmlp_backward_swiglu; FLOPs: forward 6 M H F, backward 12 M H F (dY 2, dX 4 over the
    gate and up shards, dWg 2, dWu 2, dW2 2)."""
    import torch
    import tensor_transformer_mlp_tmem_gb300 as tp

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    gated = args.variant == "train-swiglu"
    d = synth.make_swiglu_inputs(w.H, w.F, w.M, w.seed) if gated else synth.workload_inputs(w)
    dZh = synth.normal_bf16(w.seed, 60, (w.M, w.H), 1.0)

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    X = to_dev(d["X"]).view(w.B, w.S, w.H)
    W1 = to_dev(d["Wg"] if gated else d["W1"])
    W2 = to_dev(d["W2"])
    dZ = to_dev(dZh).view(w.B, w.S, w.H)
    M = w.M
    Z = torch.empty_like(X)
    Ys = torch.empty((M, w.F), dtype=torch.bfloat16, device=dev)
    As = torch.empty((M, 2 * w.F if gated else w.F), dtype=torch.bfloat16, device=dev)
    dX = torch.empty_like(X)
    f32 = torch.float32
    dW1 = torch.empty((w.H, w.F), dtype=f32, device=dev)
    db1 = torch.empty((w.F,), dtype=f32, device=dev)
    dW2 = torch.empty((w.F, w.H), dtype=f32, device=dev)
    db2 = torch.empty((w.H,), dtype=f32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    mlp = tp.TPMLP(w.H, w.F, w.k, swiglu=gated)
    if gated:
        Wu = to_dev(d["Wu"])
        dWu = torch.empty_like(dW1)
        dbu = torch.empty_like(db1)
        mlp.pack_swiglu(W1, to_dev(d["bg"]), Wu, to_dev(d["bu"]), W2, to_dev(d["b2"]))
    else:
        mlp.pack(W1, to_dev(d["b1"]), W2, to_dev(d["b2"]))
    mlp.reserve(M)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        tp.tpmlp_forward_train(mlp.ctx, X, w.B, w.S, Z, Ys, As, stream)
        if ev is not None:
            ev[1].record(stream)
        if gated:
            tp.tpmlp_backward_swiglu(mlp.ctx, dZ, X, Ys, As, W1, Wu, W2, w.B, w.S, dX, dW1, db1,
                                     dWu, dbu, dW2, db2, stream)
        else:
            tp.tpmlp_backward(mlp.ctx, dZ, X, Ys, As, W1, W2, w.B, w.S, dX, dW1, db1, dW2, db2,
                              stream)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        l2_flush(flush)
        step()
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(smi_gpu_id(local_rank))
    clocks.start()
    time.sleep(0.3)
    n0 = mlp.launches
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize(dev)
    clocks.mark_start()
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        l2_flush(flush)
        step(evs[i])
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall0
    clocks.mark_stop()
    if pg is not None:
        pg.barrier()
    launches = mlp.launches - n0
    clk = clocks.stop()
    rc, detail = mlp.status()
    if rc != tp.TPMLP_OK:
        raise RuntimeError(f"device status {detail:#x}")
    fwd = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    bwd = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    ms = fwd + bwd
    ms, fwd, bwd = max_over_ranks([ms, fwd, bwd], pg, dev)
    flops = (18 if gated else 12) * M * w.H * w.F
    peaks, peak_src = load_peaks()
    peak, regime = peak_for(peaks, t_wall)
    value = whole_job_tflops(world, flops, ms)
    bwd_tf = (12 if gated else 8) * M * w.H * w.F / (bwd * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; dZ ~ N(0,1))",
        "tokens_per_s": world * M / (ms * 1e-3),
        "peak_regime": regime, "timed_region_s": t_wall,
        "kernel_ms": {"forward_train": fwd, "backward": bwd},
        "config": workload_config(w, {"parallelism": "replicas" if world > 1 else "single GPU",
                                      "flops_per_step": flops,
                                      "step": ("forward_train + backward_swiglu (dX, dWg, dbg, dWu, "
                                               "dbu, dW2, db2)") if gated else
                                              "forward_train + backward (dX, dW1, db1, dW2, db2)"},
                                  variant="swiglu" if gated else "gelu"),
        "roofline": {"bound": "tensor",
                     "kernel": ("backward (dG/dU, dX, dWg, dWu, dW2 GEMMs + bias sums)" if gated
                                else "backward (dA, dX, dW1, dW2 GEMMs + bias sums)"),
                     "achieved": bwd_tf, "peak": peak, "unit": "TFLOP/s", "frac": bwd_tf / peak,
                     "peak_source": f"{peak_src} bf16_tflops ({regime})", "traffic": None},
        "gpu_launches": launches, "clocks": clk,
    }
    line["config"]["variant"] = args.variant
    mlp.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.barrier()
        pg.destroy_process_group()
    return 0


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.txt")


def measured_traffic(workload: str, kernel: str, build_id: str):
    """DRAM bytes per launch of `kernel` on `workload` from an ncu capture of the library build
    that is running: a line `traffic <workload> <kernel> <bytes> build <id>` of the profiles'
    traffic summary whose id equals tpmlp_build_id(). Returns (bytes or None, why)."""
    if not os.path.exists(TRAFFIC_FILE):
        return None, "no traffic summary committed"
    stale = None
    with open(TRAFFIC_FILE) as fh:
        for ln in fh:
            parts = ln.split()
            if len(parts) == 6 and parts[0] == "traffic" and parts[1] == workload \
                    and parts[2] == kernel and parts[4] == "build":
                if parts[5] != build_id:
                    stale = parts[5]
                    continue
                try:
                    return float(parts[3]), (f"ncu dram__bytes_read.sum + dram__bytes_write.sum "
                                             f"of this build ({build_id})")
                except ValueError:
                    return None, "unreadable traffic line"
    if stale:
        return None, f"the capture is of another build ({stale}); this build is {build_id}"
    return None, f"no capture of {kernel} on {workload}"


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="gpt3-175b", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--secondary", default="7b,gpt2-small,sweep-h4096:1/8/16",
                    help="other workloads timed the same way after the headline one, reported "
                         "under the line's 'secondary' key (name[:k1/k2/...], comma separated; "
                         "'' for none)")
    ap.add_argument("--k", type=int, default=None, help="override the shard count")
    ap.add_argument("--variant", default="gelu",
                    choices=["gelu", "swiglu", "block", "outproj", "qkv", "train", "train-swiglu"],
                    help="gelu: the block of the pages' Megatron figure; swiglu: the gated block; "
                         "block: Z = X + MLP(LayerNorm(X)) (LayerNorm kernel + the GeLU block "
                         "with the residual add in the second GEMM's epilogue); outproj / qkv: "
                         "the tensor-parallel attention's output (row-parallel) and Q/K/V "
                         "(column-parallel) projections on the workload's shape; train: the "
                         "training forward plus the backward pass; train-swiglu: the same for "
                         "the gated block")
    ap.add_argument("--impl", default="tpmlp", choices=["tpmlp", "reference"])
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--cpu-max-rows", type=int, default=4096)
    ap.add_argument("--reference-budget-s", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--shape", default=None, metavar="H,F,k,M",
                    help="a custom block shape instead of --workload (seeded like the named "
                         "workloads; for profiling a kernel at another shape)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.shape:
        args.secondary = ""  # a custom shape is timed alone (kernel profiling)
    try:
        parse_secondary(args.secondary)
    except ValueError as e:
        ap.error(str(e))
    w = synth.WORKLOADS[args.workload]
    if args.shape:
        try:
            H, F, k, M = (int(v) for v in args.shape.split(","))
        except ValueError:
            ap.error("--shape wants four integers H,F,k,M")
        w = synth.Workload(f"custom-h{H}-f{F}-k{k}-m{M}", 1, M, H, F, k, 7)
    if args.k is not None:
        w = synth.Workload(w.name, w.B, w.S, w.H, w.F, args.k, w.seed)
    if args.impl == "reference":
        if args.variant in ("outproj", "qkv", "train", "train-swiglu"):
            ap.error("the reference arm covers the MLP variants")
        return run_reference(args, w)
    if args.variant in ("outproj", "qkv"):
        return run_gpu_linear(args, w)
    if args.variant in ("train", "train-swiglu"):
        return run_gpu_train(args, w)
    return run_gpu(args, w)


if __name__ == "__main__":
    sys.exit(main())
