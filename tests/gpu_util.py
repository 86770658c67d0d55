"""Helpers shared by the GPU tests: bf16 bit patterns <-> CUDA tensors, error measures."""
from __future__ import annotations

import numpy as np
import torch

import synth

# Bars for the block output against the fp64 oracle (relative Frobenius error and max
# absolute error relative to max |Z_ref|), and between shard counts on the GPU.
REL_FRO_BAR = 1e-2
MAX_ABS_BAR = 3e-2
K_INVARIANCE_BAR = 2e-3


def to_dev(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """bf16 bit patterns (numpy uint16) -> bf16 CUDA tensor, same shape."""
    a = np.ascontiguousarray(bits)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def rel_fro(a: np.ndarray, ref: np.ndarray) -> float:
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(a - ref) / (den if den > 0 else 1.0))


def max_abs_rel(a: np.ndarray, ref: np.ndarray) -> float:
    m = np.max(np.abs(ref)) if ref.size else 0.0
    return float(np.max(np.abs(a - ref)) / (m if m > 0 else 1.0)) if ref.size else 0.0


def assert_close(a: np.ndarray, ref: np.ndarray, rel=REL_FRO_BAR, mx=MAX_ABS_BAR, what=""):
    r, m = rel_fro(a, ref), max_abs_rel(a, ref)
    assert r <= rel and m <= mx, f"{what}: rel_fro={r:.3e} (bar {rel}) max_abs={m:.3e} (bar {mx})"
    return r, m


class DeviceView:
    """__cuda_array_interface__ over a raw device pointer (to read library-owned buffers)."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (ptr, False), "version": 3, "strides": None}


def device_tensor(ptr: int, shape, dtype: str) -> torch.Tensor:
    typestr = {"u16": "<u2", "f32": "<f4", "i16": "<i2"}[dtype]
    return torch.as_tensor(DeviceView(ptr, shape, typestr), device="cuda")


def inputs_on_device(d: dict):
    return {k: to_dev(v) for k, v in d.items()}


def f64(bits):
    return synth.bf16_to_f64(bits)
