"""tensor_transformer_mlp_tmem_gb300 -- the Megatron-style tensor-parallel MLP block on one
GB300, all k shards on one GPU, the cross-shard sum done in tensor memory.

This module is the Python binding of ``libtpmlp.so`` (include/tpmlp.h): the functions
below carry the C entry points' names and only marshal arguments (device pointers, sizes,
streams). Every step of the block runs in the library's CUDA kernels; there is no Python
or CPU fallback, and importing a function whose library is missing raises.

The block (千亿参数模型如何拆分到多张GPU上训练, "方案一"/"方案二"; 大模型分布式并行策略详解 §4.1;
AI大模型分布式训练 §2.1-2.2):  Y_i = GeLU(X W1_i + b1_i),  Z = sum_i Y_i W2_i + b2.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "TPMLP", "TpmlpError", "load_library", "library_path",
    "tpmlp_create", "tpmlp_pack_shards", "tpmlp_reserve", "tpmlp_forward", "tpmlp_forward_host",
    "tpmlp_forward_noalloc", "TPMLP_NOALLOC_SCRATCH_BYTES",
    "tpmlp_gemm1", "tpmlp_gemm2", "tpmlp_get_status", "tpmlp_packed_buffer", "tpmlp_destroy",
    "tpmlp_strerror", "tpmlp_last_error", "tpmlp_launch_count",
    "TPMLP_OK", "TPMLP_ERR_INVALID_ARG", "TPMLP_ERR_UNSUPPORTED_SHAPE", "TPMLP_ERR_NOT_PACKED",
    "TPMLP_ERR_CUDA", "TPMLP_ERR_OOM", "TPMLP_ERR_DEVICE_TIMEOUT", "TPMLP_ERR_ARCH",
    "TPMLP_ERR_MISALIGNED", "TPMLP_FLAG_Z_FP32", "TPMLP_FLAG_SINGLE_SM", "TPMLP_FLAG_SWIGLU", "TPMLP_FLAG_FIXED_ORDER", "tpmlp_pack_shards_swiglu",
    "tpmlp_set_layernorm", "tpmlp_layernorm", "tpmlp_block_forward", "tpmlp_block_forward_host",
    "tpmlp_gemm2_residual",
    "tpmlp_linear_create", "tpmlp_linear_pack", "tpmlp_linear_forward", "Linear",
    "TPMLP_LINEAR_COLUMN", "TPMLP_LINEAR_ROW", "tpmlp_forward_train", "tpmlp_backward",
    "tpmlp_backward_swiglu", "tpmlp_set_device_rates", "tpmlp_get_device_rates", "tpmlp_build_id",
    "tpmlp_forward_marked", "tpmlp_block_forward_marked", "tpmlp_forward_host_async",
    "tpmlp_block_forward_host_async", "tpmlp_host_wait",
]

TPMLP_OK = 0
TPMLP_ERR_INVALID_ARG = -1
TPMLP_ERR_UNSUPPORTED_SHAPE = -2
TPMLP_ERR_NOT_PACKED = -3
TPMLP_ERR_CUDA = -4
TPMLP_ERR_OOM = -5
TPMLP_ERR_DEVICE_TIMEOUT = -6
TPMLP_ERR_ARCH = -7
TPMLP_ERR_MISALIGNED = -8
TPMLP_FLAG_Z_FP32 = 0x1
TPMLP_FLAG_SINGLE_SM = 0x2
TPMLP_FLAG_SWIGLU = 0x4
TPMLP_FLAG_FIXED_ORDER = 0x8
TPMLP_LINEAR_COLUMN = 0
TPMLP_LINEAR_ROW = 1
TPMLP_NOALLOC_SCRATCH_BYTES = 32 << 20  # the library's fixed scratch for tpmlp_forward_noalloc

_PKG = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    return os.path.join(_PKG, "libtpmlp.so")


class TpmlpError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: {tpmlp_strerror(status)} ({status})"
        if detail:
            msg += f": {detail}"
        super().__init__(msg)


_lib = None


def load_library() -> ctypes.CDLL:
    """Load libtpmlp.so (built in-tree by ``__graft_entry__.build()``). Raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built: run `python -c 'import __graft_entry__ as g; "
                           f"g.build()'` (nvcc, sm_103a). There is no fallback path.")
    lib = ctypes.CDLL(path)
    vp, i64, i32, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32
    sig = {
        "tpmlp_create": ([ctypes.POINTER(vp), i64, i64, i32, u32], ctypes.c_int),
        "tpmlp_pack_shards": ([vp, vp, vp, vp, vp, vp], ctypes.c_int),
        "tpmlp_pack_shards_swiglu": ([vp, vp, vp, vp, vp, vp, vp, vp], ctypes.c_int),
        "tpmlp_reserve": ([vp, i64], ctypes.c_int),
        "tpmlp_forward": ([vp, vp, i64, i64, vp, vp], ctypes.c_int),
        "tpmlp_forward_host": ([vp, vp, i64, i64, vp, vp], ctypes.c_int),
        "tpmlp_forward_host_async": ([vp, vp, i64, i64, vp, vp], ctypes.c_int),
        "tpmlp_block_forward_host_async": ([vp, vp, i64, i64, vp, vp], ctypes.c_int),
        "tpmlp_host_wait": ([vp], ctypes.c_int),
        "tpmlp_forward_marked": ([vp, vp, i64, i64, vp, vp, vp], ctypes.c_int),
        "tpmlp_block_forward_marked": ([vp, vp, i64, i64, vp, vp, vp, vp], ctypes.c_int),
        "tpmlp_forward_noalloc": ([vp, vp, i64, i64, vp, vp], ctypes.c_int),
        "tpmlp_set_layernorm": ([vp, vp, vp, ctypes.c_float, vp], ctypes.c_int),
        "tpmlp_layernorm": ([vp, vp, i64, vp, vp], ctypes.c_int),
        "tpmlp_block_forward": ([vp, vp, i64, i64, vp, vp], ctypes.c_int),
        "tpmlp_block_forward_host": ([vp, vp, i64, i64, vp, vp], ctypes.c_int),
        "tpmlp_gemm1": ([vp, vp, i64, vp, vp], ctypes.c_int),
        "tpmlp_gemm2": ([vp, vp, i64, vp, vp], ctypes.c_int),
        "tpmlp_gemm2_residual": ([vp, vp, i64, vp, vp, vp], ctypes.c_int),
        "tpmlp_get_status": ([vp, vp, ctypes.POINTER(i32)], ctypes.c_int),
        "tpmlp_packed_buffer": ([vp, i32, ctypes.POINTER(vp), ctypes.POINTER(i64)], ctypes.c_int),
        "tpmlp_linear_create": ([ctypes.POINTER(vp), i32, i64, i64, i32, u32], ctypes.c_int),
        "tpmlp_linear_pack": ([vp, vp, vp, vp], ctypes.c_int),
        "tpmlp_linear_forward": ([vp, vp, i64, vp, vp], ctypes.c_int),
        "tpmlp_forward_train": ([vp, vp, i64, i64, vp, vp, vp, vp], ctypes.c_int),
        "tpmlp_backward_swiglu": ([vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, vp, vp, vp, vp,
                                   vp, vp, vp, vp], ctypes.c_int),
        "tpmlp_backward": ([vp, vp, vp, vp, vp, vp, vp, i64, i64, vp, vp, vp, vp, vp, vp],
                           ctypes.c_int),
        "tpmlp_destroy": ([vp], None),
        "tpmlp_strerror": ([ctypes.c_int], ctypes.c_char_p),
        "tpmlp_last_error": ([vp], ctypes.c_char_p),
        "tpmlp_launch_count": ([vp], i64),
        "tpmlp_set_device_rates": ([vp, ctypes.c_double, ctypes.c_double, ctypes.c_double],
                                   ctypes.c_int),
        "tpmlp_get_device_rates": ([vp, ctypes.POINTER(ctypes.c_double),
                                    ctypes.POINTER(ctypes.c_double),
                                    ctypes.POINTER(ctypes.c_double)], ctypes.c_int),
        "tpmlp_build_id": ([], ctypes.c_char_p),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


# ------------------------------------------------------------------ marshalling helpers
def _ptr(x) -> int | None:
    """Device/host address of a torch tensor, numpy array, ctypes object or int."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    if hasattr(x, "ctypes"):
        return int(x.ctypes.data)
    if isinstance(x, ctypes.c_void_p):
        return x.value
    raise TypeError(f"cannot take the address of {type(x).__name__}")


def _stream(s) -> int | None:
    if s is None:
        try:
            import torch
            if torch.cuda.is_available() and torch.cuda.is_initialized():
                return int(torch.cuda.current_stream().cuda_stream) or None
        except Exception:  # torch absent: the legacy default stream
            pass
        return None
    if isinstance(s, int):
        return s or None
    if hasattr(s, "cuda_stream"):
        return int(s.cuda_stream) or None
    raise TypeError("stream must be a torch.cuda.Stream, an int handle or None")


def _check(rc: int, where: str, ctx=None):
    if rc != TPMLP_OK:
        detail = tpmlp_last_error(ctx) if ctx is not None else ""
        raise TpmlpError(rc, where, detail)


# ------------------------------------------------------------------ C entry points
def tpmlp_create(H: int, F: int, k: int, flags: int = 0) -> int:
    out = ctypes.c_void_p()
    _check(load_library().tpmlp_create(ctypes.byref(out), H, F, k, flags), "tpmlp_create")
    return out.value


def tpmlp_pack_shards(ctx: int, W1, b1, W2, b2, stream=None) -> None:
    _check(load_library().tpmlp_pack_shards(ctx, _ptr(W1), _ptr(b1), _ptr(W2), _ptr(b2),
                                            _stream(stream)), "tpmlp_pack_shards", ctx)


def tpmlp_pack_shards_swiglu(ctx: int, Wg, bg, Wu, bu, W2, b2, stream=None) -> None:
    _check(load_library().tpmlp_pack_shards_swiglu(ctx, _ptr(Wg), _ptr(bg), _ptr(Wu), _ptr(bu),
                                                   _ptr(W2), _ptr(b2), _stream(stream)),
           "tpmlp_pack_shards_swiglu", ctx)


def tpmlp_reserve(ctx: int, max_tokens: int) -> None:
    _check(load_library().tpmlp_reserve(ctx, max_tokens), "tpmlp_reserve", ctx)


def tpmlp_forward(ctx: int, X, B: int, S: int, Z, stream=None) -> None:
    _check(load_library().tpmlp_forward(ctx, _ptr(X), B, S, _ptr(Z), _stream(stream)),
           "tpmlp_forward", ctx)


def _event(ev) -> int:
    """cudaEvent_t handle of a torch.cuda.Event (created if it was not yet) or an int."""
    if isinstance(ev, int):
        return ev
    h = int(getattr(ev, "cuda_event", 0) or 0)
    if not h:
        ev.record()  # torch creates its event on the first record
        h = int(ev.cuda_event)
    return h


def tpmlp_forward_marked(ctx: int, X, B: int, S: int, Z, after_gemm1, stream=None) -> None:
    """tpmlp_forward, recording `after_gemm1` (a torch.cuda.Event or a raw handle) between the
    two kernel launches."""
    _check(load_library().tpmlp_forward_marked(ctx, _ptr(X), B, S, _ptr(Z), _event(after_gemm1),
                                               _stream(stream)), "tpmlp_forward_marked", ctx)


def tpmlp_block_forward_marked(ctx: int, X, B: int, S: int, Z, after_layernorm, after_gemm1,
                               stream=None) -> None:
    _check(load_library().tpmlp_block_forward_marked(ctx, _ptr(X), B, S, _ptr(Z),
                                                     _event(after_layernorm), _event(after_gemm1),
                                                     _stream(stream)),
           "tpmlp_block_forward_marked", ctx)


def tpmlp_forward_host(ctx: int, X_host, B: int, S: int, Z_host, stream=None) -> None:
    _check(load_library().tpmlp_forward_host(ctx, _ptr(X_host), B, S, _ptr(Z_host),
                                             _stream(stream)), "tpmlp_forward_host", ctx)


def tpmlp_forward_host_async(ctx: int, X_host, B: int, S: int, Z_host, stream=None) -> None:
    """Queues the forward on host buffers and returns; X_host and Z_host (pinned torch CPU
    tensors) must stay alive and untouched until tpmlp_host_wait."""
    _check(load_library().tpmlp_forward_host_async(ctx, _ptr(X_host), B, S, _ptr(Z_host),
                                                   _stream(stream)), "tpmlp_forward_host_async", ctx)


def tpmlp_block_forward_host_async(ctx: int, X_host, B: int, S: int, Z_host, stream=None) -> None:
    _check(load_library().tpmlp_block_forward_host_async(ctx, _ptr(X_host), B, S, _ptr(Z_host),
                                                         _stream(stream)),
           "tpmlp_block_forward_host_async", ctx)


def tpmlp_host_wait(ctx: int) -> None:
    _check(load_library().tpmlp_host_wait(ctx), "tpmlp_host_wait", ctx)


def tpmlp_forward_noalloc(ctx: int, X, B: int, S: int, Z, stream=None) -> None:
    """tpmlp_forward without any allocation: Y goes to the library's fixed device array
    (B*S*F*2 <= TPMLP_NOALLOC_SCRATCH_BYTES). For callers that cannot allocate device memory
    when they run the block. Calls that overlap on the GPU share that array and race."""
    _check(load_library().tpmlp_forward_noalloc(ctx, _ptr(X), B, S, _ptr(Z), _stream(stream)),
           "tpmlp_forward_noalloc", ctx)


def tpmlp_set_layernorm(ctx: int, gamma, beta, eps: float, stream=None) -> None:
    _check(load_library().tpmlp_set_layernorm(ctx, _ptr(gamma), _ptr(beta), eps, _stream(stream)),
           "tpmlp_set_layernorm", ctx)


def tpmlp_layernorm(ctx: int, X, M: int, Xn, stream=None) -> None:
    _check(load_library().tpmlp_layernorm(ctx, _ptr(X), M, _ptr(Xn), _stream(stream)),
           "tpmlp_layernorm", ctx)


def tpmlp_block_forward(ctx: int, X, B: int, S: int, Z, stream=None) -> None:
    _check(load_library().tpmlp_block_forward(ctx, _ptr(X), B, S, _ptr(Z), _stream(stream)),
           "tpmlp_block_forward", ctx)


def tpmlp_block_forward_host(ctx: int, X_host, B: int, S: int, Z_host, stream=None) -> None:
    _check(load_library().tpmlp_block_forward_host(ctx, _ptr(X_host), B, S, _ptr(Z_host),
                                                   _stream(stream)), "tpmlp_block_forward_host", ctx)


def tpmlp_gemm1(ctx: int, X, M: int, Y, stream=None) -> None:
    _check(load_library().tpmlp_gemm1(ctx, _ptr(X), M, _ptr(Y), _stream(stream)), "tpmlp_gemm1",
           ctx)


def tpmlp_gemm2(ctx: int, Y, M: int, Z, stream=None) -> None:
    _check(load_library().tpmlp_gemm2(ctx, _ptr(Y), M, _ptr(Z), _stream(stream)), "tpmlp_gemm2",
           ctx)


def tpmlp_gemm2_residual(ctx: int, Y, M: int, Z, R, stream=None) -> None:
    _check(load_library().tpmlp_gemm2_residual(ctx, _ptr(Y), M, _ptr(Z), _ptr(R), _stream(stream)),
           "tpmlp_gemm2_residual", ctx)


def tpmlp_get_status(ctx: int, stream=None):
    """Returns (status, raw detail word); clears the device status word."""
    detail = ctypes.c_int32(0)
    rc = load_library().tpmlp_get_status(ctx, _stream(stream), ctypes.byref(detail))
    if rc not in (TPMLP_OK, TPMLP_ERR_DEVICE_TIMEOUT):
        _check(rc, "tpmlp_get_status", ctx)
    return rc, int(detail.value)


def tpmlp_packed_buffer(ctx: int, which: int):
    """(device pointer, bytes) of a packed buffer: 0 W1p, 1 W2p, 2 b1 fp32, 3 b2 fp32."""
    p = ctypes.c_void_p()
    n = ctypes.c_int64()
    _check(load_library().tpmlp_packed_buffer(ctx, which, ctypes.byref(p), ctypes.byref(n)),
           "tpmlp_packed_buffer", ctx)
    return p.value, n.value


def tpmlp_linear_create(kind: int, K: int, N: int, k: int, flags: int = 0) -> int:
    out = ctypes.c_void_p()
    _check(load_library().tpmlp_linear_create(ctypes.byref(out), kind, K, N, k, flags),
           "tpmlp_linear_create")
    return out.value


def tpmlp_linear_pack(ctx: int, W, b, stream=None) -> None:
    _check(load_library().tpmlp_linear_pack(ctx, _ptr(W), _ptr(b), _stream(stream)),
           "tpmlp_linear_pack", ctx)


def tpmlp_linear_forward(ctx: int, X, M: int, out, stream=None) -> None:
    _check(load_library().tpmlp_linear_forward(ctx, _ptr(X), M, _ptr(out), _stream(stream)),
           "tpmlp_linear_forward", ctx)


def tpmlp_forward_train(ctx: int, X, B: int, S: int, Z, Ysave, Asave, stream=None) -> None:
    _check(load_library().tpmlp_forward_train(ctx, _ptr(X), B, S, _ptr(Z), _ptr(Ysave),
                                              _ptr(Asave), _stream(stream)),
           "tpmlp_forward_train", ctx)


def tpmlp_backward(ctx: int, dZ, X, Ysave, Asave, W1, W2, B: int, S: int, dX, dW1, db1, dW2,
                   db2, stream=None) -> None:
    _check(load_library().tpmlp_backward(
        ctx, _ptr(dZ), _ptr(X), _ptr(Ysave), _ptr(Asave), _ptr(W1), _ptr(W2), B, S, _ptr(dX),
        _ptr(dW1), _ptr(db1), _ptr(dW2), _ptr(db2), _stream(stream)), "tpmlp_backward", ctx)


def tpmlp_backward_swiglu(ctx: int, dZ, X, Ysave, Asave, Wg, Wu, W2, B: int, S: int, dX, dWg,
                          dbg, dWu, dbu, dW2, db2, stream=None) -> None:
    _check(load_library().tpmlp_backward_swiglu(
        ctx, _ptr(dZ), _ptr(X), _ptr(Ysave), _ptr(Asave), _ptr(Wg), _ptr(Wu), _ptr(W2), B, S,
        _ptr(dX), _ptr(dWg), _ptr(dbg), _ptr(dWu), _ptr(dbu), _ptr(dW2), _ptr(db2),
        _stream(stream)), "tpmlp_backward_swiglu", ctx)


def tpmlp_destroy(ctx) -> None:
    load_library().tpmlp_destroy(ctx)


def tpmlp_strerror(status: int) -> str:
    return load_library().tpmlp_strerror(status).decode()


def tpmlp_last_error(ctx) -> str:
    return load_library().tpmlp_last_error(ctx).decode()


def tpmlp_launch_count(ctx) -> int:
    return int(load_library().tpmlp_launch_count(ctx))


def tpmlp_set_device_rates(ctx: int, gemm_flops: float = 0.0, dram_Bps: float = 0.0,
                           copy_Bps: float = 0.0) -> None:
    """Override the planners' rates (0 keeps a rate as it is)."""
    _check(load_library().tpmlp_set_device_rates(ctx, gemm_flops, dram_Bps, copy_Bps),
           "tpmlp_set_device_rates", ctx)


def tpmlp_get_device_rates(ctx: int):
    """(gemm_flops, dram_Bps, copy_Bps) the context's planners use."""
    g, d, c = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    _check(load_library().tpmlp_get_device_rates(ctx, ctypes.byref(g), ctypes.byref(d),
                                                 ctypes.byref(c)), "tpmlp_get_device_rates", ctx)
    return g.value, d.value, c.value


def tpmlp_build_id() -> str:
    """16 hex digits identifying the library's sources and compile flags."""
    return load_library().tpmlp_build_id().decode()


# ------------------------------------------------------------------ object wrapper
class TPMLP:
    """One block shape on the current CUDA device (torch supplies memory and streams).

        mlp = TPMLP(H, F, k)
        mlp.pack(W1, b1, W2, b2)       # bf16 CUDA tensors [H,F], [F], [F,H], [H]
        Z = mlp(X)                     # X bf16 [B, S, H] -> Z [B, S, H]
    """

    def __init__(self, H: int, F: int, k: int, z_fp32: bool = False, single_sm: bool = False,
                 swiglu: bool = False, fixed_order: bool = False):
        self.H, self.F, self.k = H, F, k
        self.z_fp32 = z_fp32
        self.swiglu = swiglu
        flags = ((TPMLP_FLAG_Z_FP32 if z_fp32 else 0) | (TPMLP_FLAG_SINGLE_SM if single_sm else 0)
                 | (TPMLP_FLAG_SWIGLU if swiglu else 0)
                 | (TPMLP_FLAG_FIXED_ORDER if fixed_order else 0))
        self.ctx = tpmlp_create(H, F, k, flags)

    def close(self):
        if getattr(self, "ctx", None):
            tpmlp_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    @staticmethod
    def _require(t, dtype, shape, what):
        import torch
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{what} must be a CUDA tensor")
        if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
            raise ValueError(f"{what}: expected contiguous {dtype} {tuple(shape)}, got "
                             f"{t.dtype} {tuple(t.shape)}")

    def pack(self, W1, b1, W2, b2, stream=None):
        import torch
        bf = torch.bfloat16
        self._require(W1, bf, (self.H, self.F), "W1")
        self._require(b1, bf, (self.F,), "b1")
        self._require(W2, bf, (self.F, self.H), "W2")
        self._require(b2, bf, (self.H,), "b2")
        tpmlp_pack_shards(self.ctx, W1, b1, W2, b2, stream)

    def pack_swiglu(self, Wg, bg, Wu, bu, W2, b2, stream=None):
        """Gated block: Y = SiLU(X Wg + bg) * (X Wu + bu), then the row-parallel W2."""
        import torch
        bf = torch.bfloat16
        for t, shape, name in ((Wg, (self.H, self.F), "Wg"), (bg, (self.F,), "bg"),
                               (Wu, (self.H, self.F), "Wu"), (bu, (self.F,), "bu"),
                               (W2, (self.F, self.H), "W2"), (b2, (self.H,), "b2")):
            self._require(t, bf, shape, name)
        tpmlp_pack_shards_swiglu(self.ctx, Wg, bg, Wu, bu, W2, b2, stream)

    def set_layernorm(self, gamma, beta, eps: float = 1e-5, stream=None):
        import torch
        self._require(gamma, torch.bfloat16, (self.H,), "gamma")
        self._require(beta, torch.bfloat16, (self.H,), "beta")
        tpmlp_set_layernorm(self.ctx, gamma, beta, eps, stream)

    def layernorm(self, X2d, Xn=None, stream=None):
        import torch
        M = X2d.shape[0]
        self._require(X2d, torch.bfloat16, (M, self.H), "X")
        if Xn is None:
            Xn = torch.empty_like(X2d)
        tpmlp_layernorm(self.ctx, X2d, M, Xn, stream)
        return Xn

    def block(self, X, Z=None, stream=None):
        """Z = X + MLP(LayerNorm(X)); pass Z=X to update the residual stream in place."""
        import torch
        B, S, H = X.shape
        self._require(X, torch.bfloat16, (B, S, self.H), "X")
        if Z is None:
            Z = torch.empty((B, S, self.H), dtype=self.out_dtype(), device=X.device)
        tpmlp_block_forward(self.ctx, X, B, S, Z, stream)
        return Z

    def forward_train(self, X, stream=None):
        """Returns (Z, Ysave, Asave); Ysave/Asave feed backward() (backward_swiglu() for a
        gated block, whose Asave is [M, 2F]: G then U)."""
        import torch
        B, S, H = X.shape
        self._require(X, torch.bfloat16, (B, S, self.H), "X")
        M = B * S
        Z = torch.empty((B, S, self.H), dtype=self.out_dtype(), device=X.device)
        Ys = torch.empty((M, self.F), dtype=torch.bfloat16, device=X.device)
        As = torch.empty((M, 2 * self.F if self.swiglu else self.F), dtype=torch.bfloat16,
                         device=X.device)
        tpmlp_forward_train(self.ctx, X, B, S, Z, Ys, As, stream)
        return Z, Ys, As

    def backward(self, dZ, X, Ysave, Asave, W1, W2, stream=None):
        """Gradients (dX, dW1, db1, dW2, db2) for upstream dZ [B, S, H]."""
        import torch
        B, S, H = X.shape
        M = B * S
        dev = X.device
        dX = torch.empty((B, S, self.H), dtype=self.out_dtype(), device=dev)
        f32 = torch.float32
        dW1 = torch.empty((self.H, self.F), dtype=f32, device=dev)
        db1 = torch.empty((self.F,), dtype=f32, device=dev)
        dW2 = torch.empty((self.F, self.H), dtype=f32, device=dev)
        db2 = torch.empty((self.H,), dtype=f32, device=dev)
        tpmlp_backward(self.ctx, dZ, X, Ysave, Asave, W1, W2, B, S, dX, dW1, db1, dW2, db2, stream)
        return dX, dW1, db1, dW2, db2

    def backward_swiglu(self, dZ, X, Ysave, Asave, Wg, Wu, W2, stream=None):
        """Gradients (dX, dWg, dbg, dWu, dbu, dW2, db2) of the gated block for upstream dZ."""
        import torch
        B, S, H = X.shape
        dev = X.device
        f32 = torch.float32
        dX = torch.empty((B, S, self.H), dtype=self.out_dtype(), device=dev)
        dWg = torch.empty((self.H, self.F), dtype=f32, device=dev)
        dWu = torch.empty((self.H, self.F), dtype=f32, device=dev)
        dbg = torch.empty((self.F,), dtype=f32, device=dev)
        dbu = torch.empty((self.F,), dtype=f32, device=dev)
        dW2 = torch.empty((self.F, self.H), dtype=f32, device=dev)
        db2 = torch.empty((self.H,), dtype=f32, device=dev)
        tpmlp_backward_swiglu(self.ctx, dZ, X, Ysave, Asave, Wg, Wu, W2, B, S, dX, dWg, dbg, dWu,
                              dbu, dW2, db2, stream)
        return dX, dWg, dbg, dWu, dbu, dW2, db2

    def reserve(self, max_tokens: int):
        tpmlp_reserve(self.ctx, max_tokens)

    def out_dtype(self):
        import torch
        return torch.float32 if self.z_fp32 else torch.bfloat16

    def forward(self, X, Z=None, stream=None):
        import torch
        if X.dim() != 3:
            raise ValueError("X must be [B, S, H]")
        B, S, H = X.shape
        self._require(X, torch.bfloat16, (B, S, self.H), "X")
        if Z is None:
            Z = torch.empty((B, S, self.H), dtype=self.out_dtype(), device=X.device)
        else:
            self._require(Z, self.out_dtype(), (B, S, self.H), "Z")
        tpmlp_forward(self.ctx, X, B, S, Z, stream)
        return Z

    __call__ = forward

    def gemm1(self, X2d, Y=None, stream=None):
        import torch
        M = X2d.shape[0]
        self._require(X2d, torch.bfloat16, (M, self.H), "X")
        if Y is None:
            Y = torch.empty((M, self.F), dtype=torch.bfloat16, device=X2d.device)
        tpmlp_gemm1(self.ctx, X2d, M, Y, stream)
        return Y

    def gemm2(self, Y, Z=None, stream=None):
        import torch
        M = Y.shape[0]
        self._require(Y, torch.bfloat16, (M, self.F), "Y")
        if Z is None:
            Z = torch.empty((M, self.H), dtype=self.out_dtype(), device=Y.device)
        tpmlp_gemm2(self.ctx, Y, M, Z, stream)
        return Z

    def status(self, stream=None):
        return tpmlp_get_status(self.ctx, stream)

    @property
    def launches(self) -> int:
        return tpmlp_launch_count(self.ctx)


class Linear:
    """A column- or row-parallel linear layer with all k shards on this GPU (the Q/K/V and
    output projections of tensor-parallel attention): out = X W + b, W [K, N].

        proj = Linear("row", K, N, k); proj.pack(W, b); out = proj(X2d)
    """

    def __init__(self, kind: str, K: int, N: int, k: int, out_fp32: bool = False,
                 single_sm: bool = False, fixed_order: bool = False):
        self.kind, self.K, self.N, self.k = kind, K, N, k
        self.out_fp32 = out_fp32
        flags = ((TPMLP_FLAG_Z_FP32 if out_fp32 else 0) | (TPMLP_FLAG_SINGLE_SM if single_sm else 0)
                 | (TPMLP_FLAG_FIXED_ORDER if fixed_order else 0))
        kid = {"column": TPMLP_LINEAR_COLUMN, "row": TPMLP_LINEAR_ROW}[kind]
        self.ctx = tpmlp_linear_create(kid, K, N, k, flags)

    def close(self):
        if getattr(self, "ctx", None):
            tpmlp_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def pack(self, W, b, stream=None):
        import torch
        TPMLP._require(W, torch.bfloat16, (self.K, self.N), "W")
        TPMLP._require(b, torch.bfloat16, (self.N,), "b")
        tpmlp_linear_pack(self.ctx, W, b, stream)

    def forward(self, X, out=None, stream=None):
        import torch
        M = X.shape[0]
        TPMLP._require(X, torch.bfloat16, (M, self.K), "X")
        if out is None:
            out = torch.empty((M, self.N), dtype=torch.float32 if self.out_fp32 else torch.bfloat16,
                              device=X.device)
        tpmlp_linear_forward(self.ctx, X, M, out, stream)
        return out

    __call__ = forward

    def status(self, stream=None):
        return tpmlp_get_status(self.ctx, stream)
