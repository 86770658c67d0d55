"""Seeded synthetic inputs for the tensor-parallel MLP block (shared by the oracle's
tests, the CUDA path's tests and the benchmark).

Nothing here computes any part of the block: this module only draws X, W1, b1, W2,
b2 as bfloat16 bit patterns (numpy uint16) from a counter-based generator written in
C (``synth.c``: SplitMix64 + Box-Muller, rounded once to bf16 with ties-to-even).

Workloads follow the shapes the pages use for the MLP block: X is (B, S, H), the
first weight is (H, 4H) and the second is (4H, H) (大模型分布式并行策略详解 §4.1;
AI大模型分布式训练 §2.1-2.2). Weights are drawn with variance 1/fan_in (fan_in = H for
W1, F for W2), X with unit variance, biases with standard deviation 0.02.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "_synth.so")

STREAM_X, STREAM_W1, STREAM_B1, STREAM_W2, STREAM_B2 = 0, 1, 2, 3, 4
STREAM_WU, STREAM_BU = 5, 6  # the up projection of the gated (SwiGLU) block


def build(force: bool = False) -> str:
    """Compile synth.c into _synth.so next to it (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC,
                               "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, i64, f64 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double
        vp = ctypes.c_void_p
        lib.synth_normal_bf16.argtypes = [u64, u64, f64, f64, i64, i64, vp]
        lib.synth_normal_bf16.restype = None
        lib.synth_normal_f64.argtypes = [u64, u64, f64, f64, i64, i64, vp]
        lib.synth_normal_f64.restype = None
        lib.synth_round_bf16.argtypes = [vp, i64, vp]
        lib.synth_round_bf16.restype = None
        lib.synth_mix64.argtypes = [u64]
        lib.synth_mix64.restype = u64
        lib.synth_threads.argtypes = []
        lib.synth_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def normal_bf16(seed: int, stream: int, shape, std: float, mean: float = 0.0,
                first: int = 0) -> np.ndarray:
    """Draw prod(shape) values ~ N(mean, std^2) as bf16 bit patterns (uint16)."""
    n = int(np.prod(shape, dtype=np.int64))
    out = np.empty(n, dtype=np.uint16)
    if n:
        _load().synth_normal_bf16(seed, stream, mean, std, first, n, out.ctypes.data)
    return out.reshape(shape)


def normal_f64(seed: int, stream: int, n: int, std: float = 1.0, mean: float = 0.0,
               first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    if n:
        _load().synth_normal_f64(seed, stream, mean, std, first, n, out.ctypes.data)
    return out


def round_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().synth_round_bf16(x.ctypes.data, x.size, out.ctypes.data)
    return out


def mix64(z: int) -> int:
    return int(_load().synth_mix64(z))


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float64 exactly (bf16 is the top half of an fp32)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: X (B, S, H), W1 (H, F), W2 (F, H), k shards."""
    name: str
    B: int
    S: int
    H: int
    F: int
    k: int
    seed: int
    ks: tuple = field(default=())  # shard counts swept on identical inputs (if any)

    @property
    def M(self) -> int:
        return self.B * self.S

    @property
    def flops(self) -> int:
        """Multiply-add work of the two contractions: 2*M*H*F each."""
        return 4 * self.M * self.H * self.F


WORKLOADS = {
    "tiny": Workload("tiny", 2, 64, 256, 1024, 2, 0),
    "gpt2-small": Workload("gpt2-small", 8, 1024, 768, 3072, 4, 1),
    "7b": Workload("7b", 4, 2048, 4096, 16384, 8, 2),
    "gpt3-175b": Workload("gpt3-175b", 1, 4096, 12288, 49152, 8, 3),
    "sweep-h4096": Workload("sweep-h4096", 8, 2048, 4096, 16384, 8, 4, ks=(1, 2, 4, 8, 16)),
}


def make_inputs(H: int, F: int, M: int, seed: int, x_rows=None):
    """Draw X [M,H], W1 [H,F], b1 [F], W2 [F,H], b2 [H] as bf16 bit patterns.

    ``x_rows``: if given, only those rows of X are drawn (row r of the full X is the
    same whichever subset is requested), returned as [len(x_rows), H].
    """
    if x_rows is None:
        X = normal_bf16(seed, STREAM_X, (M, H), 1.0)
    else:
        rows = np.asarray(x_rows, dtype=np.int64)
        X = np.empty((len(rows), H), dtype=np.uint16)
        for i, r in enumerate(rows):
            X[i] = normal_bf16(seed, STREAM_X, (H,), 1.0, first=int(r) * H)
    W1 = normal_bf16(seed, STREAM_W1, (H, F), 1.0 / np.sqrt(H))
    b1 = normal_bf16(seed, STREAM_B1, (F,), 0.02)
    W2 = normal_bf16(seed, STREAM_W2, (F, H), 1.0 / np.sqrt(F))
    b2 = normal_bf16(seed, STREAM_B2, (H,), 0.02)
    return {"X": X, "W1": W1, "b1": b1, "W2": W2, "b2": b2}


def make_swiglu_inputs(H: int, F: int, M: int, seed: int, x_rows=None):
    """Gated block: X, Wg = the W1 draw, bg = the b1 draw, Wu [H,F] and bu [F] from streams of
    their own (same distributions as W1, b1), W2, b2."""
    d = make_inputs(H, F, M, seed, x_rows=x_rows)
    return {"X": d["X"], "Wg": d["W1"], "bg": d["b1"],
            "Wu": normal_bf16(seed, STREAM_WU, (H, F), 1.0 / np.sqrt(H)),
            "bu": normal_bf16(seed, STREAM_BU, (F,), 0.02),
            "W2": d["W2"], "b2": d["b2"]}


def workload_inputs(w: Workload, x_rows=None):
    return make_inputs(w.H, w.F, w.M, w.seed, x_rows=x_rows)


def sample_rows(M: int, R: int, seed: int = 12345) -> np.ndarray:
    """A fixed set of R distinct token rows: first, last, and the rest spread evenly
    with a seeded jitter (rows are independent in the block, so any subset is an
    exact check of those rows)."""
    if R >= M:
        return np.arange(M, dtype=np.int64)
    base = np.linspace(0, M - 1, R).astype(np.int64)
    rng = np.random.default_rng(seed)
    jitter = rng.integers(-(M // (2 * R)), M // (2 * R) + 1, size=R) if M // (2 * R) > 0 else 0
    rows = np.clip(base + jitter, 0, M - 1)
    rows[0], rows[-1] = 0, M - 1
    return np.unique(rows)
