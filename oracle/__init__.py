"""CPU oracle for the tensor-parallel MLP block -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this package. The CUDA library never imports, links or
calls it, and this package imports nothing from the library.

The arithmetic lives in ``tpmlp_oracle.c`` (plain fp64 loops, OpenMP over token
rows); this module only compiles it with gcc and marshals numpy arrays.

What it computes (the pages' definition of the Megatron MLP block):
  Y_i = GeLU(X W1_i + b1_i)    column shards of W1 (千亿参数模型如何拆分到多张GPU上训练,
                               "方案一：按列切分权重矩阵"; AI大模型分布式训练 §2.1)
  Z   = sum_i Y_i W2_i + b2    matching row shards of W2, summed as the All-Reduce
                               would (same page, "方案二：按行切分权重矩阵", Z = Y1V1 + Y2V2;
                               大模型分布式并行策略详解 §4.1; AI大模型分布式训练 §2.2)
with GeLU(a) = a/2 (1 + erf(a/sqrt 2)) (reading: the exact form) and b2 added once.
The layer around the block: Z = X + MLP(LayerNorm(X)) (residual of AI大模型分布式训练 §3.4,
LayerNorm on the full hidden vector before the block, 大模型分布式并行策略详解 §4.2).
The parallel linear layers on their own (the tensor-parallel attention's Q/K/V projection and
output projection, AI大模型分布式训练 §2.3): column-parallel X W + b, and row-parallel
sum_i X_i W_i + b.
The backward pass of the block (dX as a sum over shards; dW1, db1, dW2, db2).
The gated variant (gate_up_proj column-parallel, down_proj row-parallel: 大模型分布式优化技术（一）
§5.1, AI大模型分布式训练 §6.1) replaces GeLU(X W1 + b1) by SiLU(X Wg + bg) * (X Wu + bu); its
backward pass gives dX (a sum over shards of the gate and up parts), dWg, dbg, dWu, dbu, dW2, db2.

Pins (tests/test_oracle.py): identity-activation case against numpy float64 matmul,
GeLU values from the normal-CDF table and scipy's ndtr, the odd-part identity
GeLU(a) - GeLU(-a) = a, W2 = 0 and W1 = 0 special cases, a hand-summed brute-force
case (tests/golden/), the row-split sum against an unsharded product, and k-invariance.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tpmlp_oracle.c")
_LIB = os.path.join(_HERE, "_oracle.so")

ACT_GELU = 0
ACT_IDENTITY = 1


def build(force: bool = False) -> str:
    """Compile the oracle (gcc -O2, OpenMP, no FMA contraction) next to its source."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                               "-std=c11", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class Oracle:
    """ctypes view of one compiled copy of the oracle's C source."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        lib.oracle_tpmlp_f64.argtypes = [vp, i64, vp, i64, vp, vp, vp, vp, i64, i64, i32, i32,
                                         vp, vp, vp]
        lib.oracle_tpmlp_f64.restype = ctypes.c_int
        lib.oracle_gelu.argtypes = [ctypes.c_double]
        lib.oracle_gelu.restype = ctypes.c_double
        lib.oracle_tpmlp_swiglu_f64.argtypes = [vp, i64, vp, i64, vp, vp, vp, vp, vp, vp, i64, i64,
                                                i32, vp, vp]
        lib.oracle_tpmlp_swiglu_f64.restype = ctypes.c_int
        lib.oracle_silu.argtypes = [ctypes.c_double]
        lib.oracle_silu.restype = ctypes.c_double
        lib.oracle_block_f64.argtypes = [vp, i64, vp, i64, vp, vp, ctypes.c_double, vp, vp, vp, vp,
                                         i64, i64, i32, vp, vp]
        lib.oracle_block_f64.restype = ctypes.c_int
        lib.oracle_linear_f64.argtypes = [i32, vp, i64, vp, i64, vp, vp, i64, i64, i32, vp]
        lib.oracle_linear_f64.restype = ctypes.c_int
        lib.oracle_gelu_grad.argtypes = [ctypes.c_double]
        lib.oracle_gelu_grad.restype = ctypes.c_double
        lib.oracle_backward_f64.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, vp, vp, vp,
                                            vp, vp]
        lib.oracle_backward_f64.restype = ctypes.c_int
        lib.oracle_silu_grad.argtypes = [ctypes.c_double]
        lib.oracle_silu_grad.restype = ctypes.c_double
        lib.oracle_swiglu_backward_f64.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i32,
                                                   vp, vp, vp, vp, vp, vp, vp]
        lib.oracle_swiglu_backward_f64.restype = ctypes.c_int
        lib.oracle_threads.argtypes = []
        lib.oracle_threads.restype = ctypes.c_int
        self.lib = lib
        self.path = lib_path

    def threads(self) -> int:
        """OpenMP threads the oracle runs with."""
        return int(self.lib.oracle_threads())

    def gelu(self, a: float) -> float:
        return float(self.lib.oracle_gelu(float(a)))

    def tpmlp(self, X, W1, b1, W2, b2, k: int, rows=None, act: int = ACT_GELU,
              want_y: bool = False, want_partials: bool = False):
        """Evaluate the block in fp64 for the selected rows of X.

        X [x_rows, H], W1 [H, F], b1 [F], W2 [F, H], b2 [H]: bf16 bit patterns (uint16).
        rows: indices into X (default: all rows). Returns {"Z": [R,H]} plus "Y" [R,F]
        and "P" [R,k,H] (per-shard partials) when asked.
        """
        X, W1, b1, W2, b2 = (_u16(a) for a in (X, W1, b1, W2, b2))
        x_rows, H = X.shape
        H1, F = W1.shape
        if H1 != H or W2.shape != (F, H) or b1.shape != (F,) or b2.shape != (H,):
            raise ValueError("shape mismatch")
        if rows is None:
            rows_arr = None
            R = x_rows
        else:
            rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
            R = len(rows_arr)
        Z = np.empty((R, H), dtype=np.float64)
        Y = np.empty((R, F), dtype=np.float64) if want_y else None
        P = np.empty((R, k, H), dtype=np.float64) if want_partials else None
        rc = self.lib.oracle_tpmlp_f64(
            X.ctypes.data, x_rows, None if rows_arr is None else rows_arr.ctypes.data, R,
            W1.ctypes.data, b1.ctypes.data, W2.ctypes.data, b2.ctypes.data, H, F, k, act,
            Z.ctypes.data, None if Y is None else Y.ctypes.data,
            None if P is None else P.ctypes.data)
        if rc != 0:
            raise ValueError("oracle rejected its arguments (F % k, rows out of range, ...)")
        out = {"Z": Z}
        if want_y:
            out["Y"] = Y
        if want_partials:
            out["P"] = P
        return out


    def silu(self, a: float) -> float:
        return float(self.lib.oracle_silu(float(a)))

    def tpmlp_swiglu(self, X, Wg, bg, Wu, bu, W2, b2, k: int, rows=None, want_y: bool = False):
        """Gated variant: Y = SiLU(X Wg + bg) * (X Wu + bu), Z = sum_i Y_i W2_i + b2 (fp64).
        X [x_rows, H]; Wg, Wu [H, F]; bg, bu [F]; W2 [F, H]; b2 [H] (bf16 bit patterns)."""
        X, Wg, bg, Wu, bu, W2, b2 = (_u16(a) for a in (X, Wg, bg, Wu, bu, W2, b2))
        x_rows, H = X.shape
        H1, F = Wg.shape
        if (H1 != H or Wu.shape != (H, F) or W2.shape != (F, H) or bg.shape != (F,)
                or bu.shape != (F,) or b2.shape != (H,)):
            raise ValueError("shape mismatch")
        rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        R = x_rows if rows_arr is None else len(rows_arr)
        Z = np.empty((R, H), dtype=np.float64)
        Y = np.empty((R, F), dtype=np.float64) if want_y else None
        rc = self.lib.oracle_tpmlp_swiglu_f64(
            X.ctypes.data, x_rows, None if rows_arr is None else rows_arr.ctypes.data, R,
            Wg.ctypes.data, bg.ctypes.data, Wu.ctypes.data, bu.ctypes.data, W2.ctypes.data,
            b2.ctypes.data, H, F, k, Z.ctypes.data, None if Y is None else Y.ctypes.data)
        if rc != 0:
            raise ValueError("oracle rejected its arguments (F % k, rows out of range, ...)")
        out = {"Z": Z}
        if want_y:
            out["Y"] = Y
        return out


    def block(self, X, gamma, beta, eps: float, W1, b1, W2, b2, k: int, rows=None,
              want_xn: bool = False):
        """Pre-LayerNorm sub-layer Z = X + MLP(LN(X)) in fp64 (gamma, beta [H] bf16)."""
        X, gamma, beta, W1, b1, W2, b2 = (_u16(a) for a in (X, gamma, beta, W1, b1, W2, b2))
        x_rows, H = X.shape
        F = W1.shape[1]
        if (W1.shape != (H, F) or W2.shape != (F, H) or gamma.shape != (H,) or beta.shape != (H,)
                or b1.shape != (F,) or b2.shape != (H,)):
            raise ValueError("shape mismatch")
        rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        R = x_rows if rows_arr is None else len(rows_arr)
        Z = np.empty((R, H), dtype=np.float64)
        Xn = np.empty((R, H), dtype=np.float64) if want_xn else None
        rc = self.lib.oracle_block_f64(
            X.ctypes.data, x_rows, None if rows_arr is None else rows_arr.ctypes.data, R,
            gamma.ctypes.data, beta.ctypes.data, float(eps), W1.ctypes.data, b1.ctypes.data,
            W2.ctypes.data, b2.ctypes.data, H, F, k, Z.ctypes.data,
            None if Xn is None else Xn.ctypes.data)
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        out = {"Z": Z}
        if want_xn:
            out["Xn"] = Xn
        return out


    def linear(self, kind: str, X, W, b, k: int, rows=None):
        """Parallel linear layer in fp64: kind "column" (W split by columns, outputs
        concatenated) or "row" (W split by rows, partials summed). X [x_rows, K], W [K, N]."""
        X, W, b = (_u16(a) for a in (X, W, b))
        x_rows, K = X.shape
        if W.shape[0] != K or b.shape != (W.shape[1],):
            raise ValueError("shape mismatch")
        N = W.shape[1]
        rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        R = x_rows if rows_arr is None else len(rows_arr)
        out = np.empty((R, N), dtype=np.float64)
        rc = self.lib.oracle_linear_f64({"column": 0, "row": 1}[kind], X.ctypes.data, x_rows,
                                        None if rows_arr is None else rows_arr.ctypes.data, R,
                                        W.ctypes.data, b.ctypes.data, K, N, k, out.ctypes.data)
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        return out


    def gelu_grad(self, a: float) -> float:
        return float(self.lib.oracle_gelu_grad(float(a)))

    def backward(self, X, W1, b1, W2, dZ, k: int):
        """Gradients of the block for upstream dZ [M, H]: dict of dX [M,H], dW1 [H,F],
        db1 [F], dW2 [F,H], db2 [H] (fp64)."""
        X, W1, b1, W2, dZ = (_u16(a) for a in (X, W1, b1, W2, dZ))
        M, H = X.shape
        F = W1.shape[1]
        if W1.shape != (H, F) or W2.shape != (F, H) or b1.shape != (F,) or dZ.shape != (M, H):
            raise ValueError("shape mismatch")
        out = {"dX": np.empty((M, H)), "dW1": np.empty((H, F)), "db1": np.empty(F),
               "dW2": np.empty((F, H)), "db2": np.empty(H)}
        rc = self.lib.oracle_backward_f64(
            X.ctypes.data, W1.ctypes.data, b1.ctypes.data, W2.ctypes.data, dZ.ctypes.data, M, H,
            F, k, out["dX"].ctypes.data, out["dW1"].ctypes.data, out["db1"].ctypes.data,
            out["dW2"].ctypes.data, out["db2"].ctypes.data)
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        return out

    def silu_grad(self, g: float) -> float:
        return float(self.lib.oracle_silu_grad(float(g)))

    def swiglu_backward(self, X, Wg, bg, Wu, bu, W2, dZ, k: int):
        """Gradients of the gated block for upstream dZ [M, H]: dict of dX [M,H], dWg [H,F],
        dbg [F], dWu [H,F], dbu [F], dW2 [F,H], db2 [H] (fp64)."""
        X, Wg, bg, Wu, bu, W2, dZ = (_u16(a) for a in (X, Wg, bg, Wu, bu, W2, dZ))
        M, H = X.shape
        F = Wg.shape[1]
        if (Wg.shape != (H, F) or Wu.shape != (H, F) or W2.shape != (F, H) or bg.shape != (F,)
                or bu.shape != (F,) or dZ.shape != (M, H)):
            raise ValueError("shape mismatch")
        out = {"dX": np.empty((M, H)), "dWg": np.empty((H, F)), "dbg": np.empty(F),
               "dWu": np.empty((H, F)), "dbu": np.empty(F), "dW2": np.empty((F, H)),
               "db2": np.empty(H)}
        rc = self.lib.oracle_swiglu_backward_f64(
            X.ctypes.data, Wg.ctypes.data, bg.ctypes.data, Wu.ctypes.data, bu.ctypes.data,
            W2.ctypes.data, dZ.ctypes.data, M, H, F, k,
            *(out[n].ctypes.data for n in ("dX", "dWg", "dbg", "dWu", "dbu", "dW2", "db2")))
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        return out


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (numpy uint16)")
    return a


def compile_source(source_text: str, out_path: str) -> Oracle:
    """Compile a (possibly edited) copy of the oracle source; used by the tests that
    plant mistakes in the oracle to show that its pins catch them."""
    src = out_path + ".c"
    with open(src, "w") as fh:
        fh.write(source_text)
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                           "-std=c11", src, "-o", out_path, "-lm"])
    return Oracle(out_path)


def source() -> str:
    with open(_SRC) as fh:
        return fh.read()


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def threads() -> int:
    return default().threads()


def gelu(a: float) -> float:
    return default().gelu(a)


def tpmlp(X, W1, b1, W2, b2, k: int, rows=None, act: int = ACT_GELU, want_y: bool = False,
          want_partials: bool = False):
    return default().tpmlp(X, W1, b1, W2, b2, k, rows=rows, act=act, want_y=want_y,
                           want_partials=want_partials)


def silu(a: float) -> float:
    return default().silu(a)


def tpmlp_swiglu(X, Wg, bg, Wu, bu, W2, b2, k: int, rows=None, want_y: bool = False):
    return default().tpmlp_swiglu(X, Wg, bg, Wu, bu, W2, b2, k, rows=rows, want_y=want_y)


def block(X, gamma, beta, eps, W1, b1, W2, b2, k: int, rows=None, want_xn: bool = False):
    return default().block(X, gamma, beta, eps, W1, b1, W2, b2, k, rows=rows, want_xn=want_xn)


def linear(kind: str, X, W, b, k: int, rows=None):
    return default().linear(kind, X, W, b, k, rows=rows)


def gelu_grad(a: float) -> float:
    return default().gelu_grad(a)


def backward(X, W1, b1, W2, dZ, k: int):
    return default().backward(X, W1, b1, W2, dZ, k)


def silu_grad(g: float) -> float:
    return default().silu_grad(g)


def swiglu_backward(X, Wg, bg, Wu, bu, W2, dZ, k: int):
    return default().swiglu_backward(X, Wg, bg, Wu, bu, W2, dZ, k)
