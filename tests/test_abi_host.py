"""The C-ABI library loads and exports every entry point include/tpmlp.h declares; host
validation rejects bad arguments before any device work (no GPU needed)."""
import ctypes
import os
import re

import pytest

import tensor_transformer_mlp_tmem_gb300 as tp
from tensor_transformer_mlp_tmem_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tpmlp.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return tp.load_library()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"TPMLP_API\s+[\w\s\*]*?\b(tpmlp_\w+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_symbols()
    for must in ("tpmlp_create", "tpmlp_pack_shards", "tpmlp_forward", "tpmlp_destroy"):
        assert must in names
    assert len(names) >= 13


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), f"{name} declared in tpmlp.h but not exported"


def test_library_exports_nothing_else(lib):
    # hidden visibility: only the declared entry points are dynamic symbols
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", tp.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = sorted({ln.split()[-1] for ln in out.splitlines() if " T " in ln})
    tpmlp_syms = [s for s in exported if s.startswith("tpmlp_")]
    assert tpmlp_syms == declared_symbols()


def test_strerror_covers_every_status(lib):
    for st in range(0, -9, -1):
        s = tp.tpmlp_strerror(st)
        assert s and s != "unknown status"
    assert tp.tpmlp_strerror(-99) == "unknown status"


def test_create_rejects_bad_arguments_before_device_work(lib):
    out = ctypes.c_void_p()
    assert lib.tpmlp_create(None, 256, 1024, 2, 0) == tp.TPMLP_ERR_INVALID_ARG
    assert lib.tpmlp_create(ctypes.byref(out), 0, 1024, 2, 0) == tp.TPMLP_ERR_INVALID_ARG
    assert lib.tpmlp_create(ctypes.byref(out), 256, 1024, 0, 0) == tp.TPMLP_ERR_INVALID_ARG
    assert lib.tpmlp_create(ctypes.byref(out), 256, 1024, 2, 0x80) == tp.TPMLP_ERR_INVALID_ARG
    # F % k != 0, shard width not a multiple of 64, H not a multiple of 64
    assert lib.tpmlp_create(ctypes.byref(out), 256, 1024, 3, 0) == tp.TPMLP_ERR_UNSUPPORTED_SHAPE
    assert lib.tpmlp_create(ctypes.byref(out), 256, 1024, 32, 0) == tp.TPMLP_ERR_UNSUPPORTED_SHAPE
    assert lib.tpmlp_create(ctypes.byref(out), 200, 1024, 2, 0) == tp.TPMLP_ERR_UNSUPPORTED_SHAPE
    assert lib.tpmlp_create(ctypes.byref(out), 256, 1000, 2, 0) == tp.TPMLP_ERR_UNSUPPORTED_SHAPE
    assert out.value is None


def test_null_context_everywhere(lib):
    INV = tp.TPMLP_ERR_INVALID_ARG
    assert lib.tpmlp_pack_shards(None, 16, 16, 16, 16, None) == INV
    assert lib.tpmlp_forward(None, 16, 1, 1, 16, None) == INV
    assert lib.tpmlp_forward_host(None, 16, 1, 1, 16, None) == INV
    assert lib.tpmlp_forward_host_async(None, 16, 1, 1, 16, None) == INV
    assert lib.tpmlp_block_forward_host_async(None, 16, 1, 1, 16, None) == INV
    assert lib.tpmlp_host_wait(None) == INV
    assert lib.tpmlp_gemm1(None, 16, 1, 16, None) == INV
    assert lib.tpmlp_gemm2(None, 16, 1, 16, None) == INV
    assert lib.tpmlp_reserve(None, 1) == INV
    assert lib.tpmlp_get_status(None, None, None) == INV
    p, n = ctypes.c_void_p(), ctypes.c_int64()
    assert lib.tpmlp_packed_buffer(None, 0, ctypes.byref(p), ctypes.byref(n)) == INV
    lib.tpmlp_destroy(None)  # no-op
    assert tp.tpmlp_last_error(None) == ""
    assert tp.tpmlp_launch_count(None) == 0


def test_binding_names_match_c_abi():
    for name in declared_symbols():
        assert hasattr(tp, name), f"binding lacks {name}"


# ------------------------------------------------------------------ device checks (test build)
@pytest.fixture(scope="module")
def hooks(tmp_path_factory):
    """A test build (-DTPMLP_TEST_HOOKS) that can make contexts holding no device memory,
    recorded on any device index, and substitute the current-device query: the device check
    of every entry point runs on a machine without a GPU."""
    path = _build.build(out=str(tmp_path_factory.mktemp("hooks") / "libtpmlp_hooks.so"),
                        extra_flags=["-DTPMLP_TEST_HOOKS"])
    h = ctypes.CDLL(path)
    vp, i64, i32, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32
    h.tpmlp_test_host_context.argtypes = [i64, i64, i32, i32, i32, i32, u32]
    h.tpmlp_test_host_context.restype = vp
    h.tpmlp_test_set_current_device.argtypes = [i32]
    h.tpmlp_last_error.argtypes = [vp]
    h.tpmlp_last_error.restype = ctypes.c_char_p
    h.tpmlp_launch_count.argtypes = [vp]
    h.tpmlp_launch_count.restype = i64
    h.tpmlp_destroy.argtypes = [vp]
    h.tpmlp_set_device_rates.argtypes = [vp, ctypes.c_double, ctypes.c_double, ctypes.c_double]
    h.tpmlp_get_device_rates.argtypes = [vp] + [ctypes.POINTER(ctypes.c_double)] * 3
    yield h
    h.tpmlp_test_set_current_device(-1)


BLOCK_CALLS = {
    # entry point -> arguments after the context (16: a non-null, 16-byte aligned address)
    "tpmlp_pack_shards": (16, 16, 16, 16, None),
    "tpmlp_reserve": (1024,),
    "tpmlp_forward": (16, 1, 64, 16, None),
    "tpmlp_forward_host": (16, 1, 64, 16, None),
    "tpmlp_forward_host_async": (16, 1, 64, 16, None),
    "tpmlp_host_wait": (),
    "tpmlp_forward_noalloc": (16, 1, 64, 16, None),
    "tpmlp_forward_marked": (16, 1, 64, 16, 16, None),
    "tpmlp_block_forward_marked": (16, 1, 64, 16, 16, 16, None),
    "tpmlp_gemm1": (16, 64, 16, None),
    "tpmlp_gemm2": (16, 64, 16, None),
    "tpmlp_gemm2_residual": (16, 64, 16, 16, None),
    "tpmlp_set_layernorm": (16, 16, ctypes.c_float(1e-5), None),
    "tpmlp_layernorm": (16, 64, 16, None),
    "tpmlp_block_forward": (16, 1, 64, 16, None),
    "tpmlp_block_forward_host": (16, 1, 64, 16, None),
    "tpmlp_block_forward_host_async": (16, 1, 64, 16, None),
    "tpmlp_forward_train": (16, 1, 64, 16, 16, 16, None),
    "tpmlp_backward": (16, 16, 16, 16, 16, 16, 1, 64, 16, 16, 16, 16, 16, None),
    "tpmlp_get_status": (None, None),
}
GATED_CALLS = {
    "tpmlp_pack_shards_swiglu": (16, 16, 16, 16, 16, 16, None),
    "tpmlp_backward_swiglu": (16, 16, 16, 16, 16, 16, 16, 1, 64, 16, 16, 16, 16, 16, 16, 16,
                              None),
}
LINEAR_CALLS = {
    "tpmlp_linear_pack": (16, 16, None),
    "tpmlp_linear_forward": (16, 64, 16, None),
}


def call(h, name, ctx, args):
    fn = getattr(h, name)
    fn.restype = ctypes.c_int
    conv = []
    for a in args:
        if isinstance(a, ctypes.c_float):
            conv.append(a)
        elif a is None:
            conv.append(ctypes.c_void_p(None))
        else:
            conv.append(ctypes.c_int64(a) if not isinstance(a, ctypes._SimpleCData) else a)
    return fn(ctypes.c_void_p(ctx), *conv)


@pytest.mark.parametrize("kind,flags,calls", [(0, 0, BLOCK_CALLS), (0, 0x4, GATED_CALLS),
                                              (1, 0, LINEAR_CALLS), (2, 0, LINEAR_CALLS)],
                         ids=["block", "gated", "column", "row"])
def test_every_entry_point_checks_the_current_device(hooks, kind, flags, calls):
    """A context of device 3 called while device 0 is current: every entry point that would
    enqueue work or touch the context's memory returns INVALID_ARG before doing anything, and
    says why; with device 3 current the same calls get past the check."""
    H, F, k = 256, 1024, 4
    ctx = hooks.tpmlp_test_host_context(H, F, k, 3, kind, 1, flags)
    assert ctx
    try:
        hooks.tpmlp_test_set_current_device(0)
        for name, args in calls.items():
            assert call(hooks, name, ctx, args) == tp.TPMLP_ERR_INVALID_ARG, name
            msg = hooks.tpmlp_last_error(ctx).decode()
            assert "device 3" in msg and "device 0" in msg, (name, msg)
        assert hooks.tpmlp_launch_count(ctx) == 0
        # the right device current: an empty batch is a no-op again
        hooks.tpmlp_test_set_current_device(3)
        if kind == 0 and not flags:
            assert call(hooks, "tpmlp_forward", ctx, (16, 0, 64, 16, None)) == tp.TPMLP_OK
            assert call(hooks, "tpmlp_forward_noalloc", ctx, (16, 0, 64, 16, None)) == tp.TPMLP_OK
            assert call(hooks, "tpmlp_gemm1", ctx, (16, 0, 16, None)) == tp.TPMLP_OK
            assert call(hooks, "tpmlp_forward_host_async", ctx, (16, 0, 64, 16, None)) == tp.TPMLP_OK
            assert call(hooks, "tpmlp_host_wait", ctx, ()) == tp.TPMLP_OK  # nothing queued
        if kind != 0:
            assert call(hooks, "tpmlp_linear_forward", ctx, (16, 0, 16, None)) == tp.TPMLP_OK
        assert hooks.tpmlp_launch_count(ctx) == 0
    finally:
        hooks.tpmlp_test_set_current_device(-1)
        hooks.tpmlp_destroy(ctypes.c_void_p(ctx))


def test_unpacked_context_on_its_device(hooks):
    """With the device current, the next check applies: weights not packed."""
    ctx = hooks.tpmlp_test_host_context(256, 1024, 4, 2, 0, 0, 0)
    try:
        hooks.tpmlp_test_set_current_device(2)
        assert call(hooks, "tpmlp_forward", ctx, (16, 1, 64, 16, None)) == tp.TPMLP_ERR_NOT_PACKED
    finally:
        hooks.tpmlp_test_set_current_device(-1)
        hooks.tpmlp_destroy(ctypes.c_void_p(ctx))


def test_device_rates_set_and_get(hooks):
    ctx = hooks.tpmlp_test_host_context(256, 1024, 4, 0, 0, 1, 0)
    try:
        vals = [ctypes.c_double() for _ in range(3)]
        refs = [ctypes.byref(v) for v in vals]
        assert hooks.tpmlp_get_device_rates(ctypes.c_void_p(ctx), *refs) == tp.TPMLP_OK
        g0, d0, c0 = (v.value for v in vals)
        assert g0 == pytest.approx(152 * 8192 * 2.07e9 * 0.67) and d0 > 1e12 and c0 == 168e9
        # 0 keeps a rate; a negative or NaN rate is rejected and changes nothing
        assert hooks.tpmlp_set_device_rates(ctypes.c_void_p(ctx), 2e15, 0.0, 100e9) == tp.TPMLP_OK
        assert hooks.tpmlp_set_device_rates(ctypes.c_void_p(ctx), -1.0, 0.0, 0.0) == \
            tp.TPMLP_ERR_INVALID_ARG
        assert hooks.tpmlp_set_device_rates(ctypes.c_void_p(ctx), float("nan"), 0.0, 0.0) == \
            tp.TPMLP_ERR_INVALID_ARG
        assert hooks.tpmlp_get_device_rates(ctypes.c_void_p(ctx), *refs) == tp.TPMLP_OK
        assert (vals[0].value, vals[1].value, vals[2].value) == (2e15, d0, 100e9)
        assert hooks.tpmlp_set_device_rates(None, 1.0, 1.0, 1.0) == tp.TPMLP_ERR_INVALID_ARG
    finally:
        hooks.tpmlp_destroy(ctypes.c_void_p(ctx))


def test_build_id_names_the_sources(lib):
    """The running library's id is the hash of the sources and flags it was built from."""
    bid = tp.tpmlp_build_id()
    assert re.fullmatch(r"[0-9a-f]{16}", bid)
    assert bid == _build.source_hash()
