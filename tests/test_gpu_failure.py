"""Failure detection without a GPU fault: a test build of the library whose TMA producer
never fills one pipeline stage (in the CTA-pair kernel: rank 0 never arms it, while its
peer's copies still land). The MMA warp's bounded wait on that stage runs out after
about a second; the kernel records where in the device status word, drains what it has in
flight, frees its tensor memory and returns. The host reads TPMLP_ERR_DEVICE_TIMEOUT and the
CUDA context stays usable (the regular library still computes the right answer afterwards).

A second test build never announces a partial sum of the split reduction: the pair that owns
the tile waits for a flag that nothing sets, gives up after about a second and reports the
split-reduction wait site."""
import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
import synth
import tensor_transformer_mlp_tmem_gb300 as tp
from tensor_transformer_mlp_tmem_gb300 import _build
from gpu_util import assert_close, inputs_on_device, to_dev, to_f64

pytestmark = pytest.mark.gpu

GEMM1_MMA_FULL_WAIT = (1 << 8) | 3  # (mode << 8) | wait site, as the kernel records it
GEMM1_PRODUCER_WAIT = (1 << 8) | 1  # the producer's wait for the stage that is never freed
PAIR = 0x80                         # set by the CTA-pair kernel


@pytest.fixture(scope="module")
def stall_lib(tmp_path_factory):
    return _build.build(out=str(tmp_path_factory.mktemp("stall") / "libtpmlp_stall.so"),
                        extra_flags=["-DTPMLP_TEST_SKIP_STAGE=5"])


@pytest.mark.parametrize("single_sm", [True, False], ids=["single-SM", "CTA-pair"])
def test_pipeline_wait_runs_out_and_is_reported(lib, stall_lib, single_sm):
    dbg = ctypes.CDLL(stall_lib)
    vp, i64, i32, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32
    dbg.tpmlp_create.argtypes = [ctypes.POINTER(vp), i64, i64, i32, u32]
    dbg.tpmlp_pack_shards.argtypes = [vp] * 6
    dbg.tpmlp_gemm1.argtypes = [vp, vp, i64, vp, vp]
    dbg.tpmlp_get_status.argtypes = [vp, vp, ctypes.POINTER(i32)]
    dbg.tpmlp_destroy.argtypes = [vp]

    H, F, k, M = 1024, 1024, 2, 256  # 16 reduction blocks per tile: stage 5 is reached
    d = synth.make_inputs(H, F, M, 191)
    dd = inputs_on_device(d)
    Y = torch.empty((M, F), dtype=torch.bfloat16, device="cuda")
    ctx = vp()
    flags = tp.TPMLP_FLAG_SINGLE_SM if single_sm else 0
    assert dbg.tpmlp_create(ctypes.byref(ctx), H, F, k, flags) == 0
    try:
        assert dbg.tpmlp_pack_shards(ctx, dd["W1"].data_ptr(), dd["b1"].data_ptr(),
                                     dd["W2"].data_ptr(), dd["b2"].data_ptr(), None) == 0
        t0 = time.time()
        assert dbg.tpmlp_gemm1(ctx, dd["X"].data_ptr(), M, Y.data_ptr(), None) == 0
        detail = ctypes.c_int32(0)
        rc = dbg.tpmlp_get_status(ctx, None, ctypes.byref(detail))
        elapsed = time.time() - t0
        assert rc == tp.TPMLP_ERR_DEVICE_TIMEOUT
        # The MMA warp waits for the stage that is never filled; a few microseconds later the
        # producer waits for that stage to be freed. Each gives up after its own second and
        # the first to give up records its site, so either may be reported.
        pair_bit = 0 if single_sm else PAIR
        assert detail.value in (GEMM1_MMA_FULL_WAIT | pair_bit, GEMM1_PRODUCER_WAIT | pair_bit), \
            hex(detail.value)
        assert 0.5 < elapsed < 30.0
        # the status word was cleared by the read
        assert dbg.tpmlp_get_status(ctx, None, ctypes.byref(detail)) == tp.TPMLP_OK
    finally:
        dbg.tpmlp_destroy(ctx)

    torch.cuda.synchronize()  # no sticky CUDA error: the context is still usable
    with tp.TPMLP(H, F, k, single_sm=single_sm) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        Z = mlp(dd["X"].view(1, M, H))
        torch.cuda.synchronize()
        assert mlp.status()[0] == tp.TPMLP_OK
    ref = oracle.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], k)["Z"]
    assert_close(to_f64(Z.view(M, H)), ref, what="after the stalled kernel")


GEMM2_SPLIT_WAIT = (2 << 8) | PAIR | 5


@pytest.fixture(scope="module")
def silent_lib(tmp_path_factory):
    return _build.build(out=str(tmp_path_factory.mktemp("silent") / "libtpmlp_silent.so"),
                        extra_flags=["-DTPMLP_TEST_SKIP_FLAG"])


def test_split_reduction_wait_runs_out_and_is_reported(lib, silent_lib):
    dbg = ctypes.CDLL(silent_lib)
    vp, i64, i32, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32
    dbg.tpmlp_create.argtypes = [ctypes.POINTER(vp), i64, i64, i32, u32]
    dbg.tpmlp_pack_shards.argtypes = [vp] * 6
    dbg.tpmlp_gemm2.argtypes = [vp, vp, i64, vp, vp]
    dbg.tpmlp_get_status.argtypes = [vp, vp, ctypes.POINTER(i32)]
    dbg.tpmlp_destroy.argtypes = [vp]

    # the second GEMM has 10 x 10 = 100 pair tiles: one wave plus a split tail
    H, F, k, M = 2560, 1024, 2, 2560
    d = synth.make_inputs(H, F, M, 193)
    dd = inputs_on_device(d)
    Y_bits = synth.normal_bf16(193, 61, (M, F), 1.0)
    Y = to_dev(Y_bits)
    Z = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    ctx = vp()
    assert dbg.tpmlp_create(ctypes.byref(ctx), H, F, k, 0) == 0
    try:
        assert dbg.tpmlp_pack_shards(ctx, dd["W1"].data_ptr(), dd["b1"].data_ptr(),
                                     dd["W2"].data_ptr(), dd["b2"].data_ptr(), None) == 0
        t0 = time.time()
        assert dbg.tpmlp_gemm2(ctx, Y.data_ptr(), M, Z.data_ptr(), None) == 0
        detail = ctypes.c_int32(0)
        rc = dbg.tpmlp_get_status(ctx, None, ctypes.byref(detail))
        elapsed = time.time() - t0
        assert rc == tp.TPMLP_ERR_DEVICE_TIMEOUT
        assert detail.value == GEMM2_SPLIT_WAIT, hex(detail.value)
        assert 0.5 < elapsed < 30.0
    finally:
        dbg.tpmlp_destroy(ctx)

    torch.cuda.synchronize()  # the context is still usable
    with tp.TPMLP(H, F, k) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        Z = mlp.gemm2(Y)
        torch.cuda.synchronize()
        assert mlp.status()[0] == tp.TPMLP_OK
    rows = synth.sample_rows(M, 16)
    ref = oracle.linear("row", Y_bits, d["W2"], d["b2"], k, rows=rows)
    assert_close(to_f64(Z)[rows], ref, what="second GEMM after the silent partial")
