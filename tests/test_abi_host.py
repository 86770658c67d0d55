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
