"""Failure detection without a GPU fault: a test build of the library whose TMA producer
never fills one pipeline stage (in the CTA-pair kernel: rank 0 never arms it, while its
peer's copies still land). The MMA warp's bounded wait on that stage runs out after
about a second; the kernel records where in the device status word, drains what it has in
flight, frees its tensor memory and returns. The host reads TPMLP_ERR_DEVICE_TIMEOUT and the
CUDA context stays usable (the regular library still computes the right answer afterwards)."""
import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
import synth
import tensor_transformer_mlp_tmem_gb300 as tp
from tensor_transformer_mlp_tmem_gb300 import _build
from gpu_util import assert_close, inputs_on_device, to_f64

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

    # 16 reduction blocks per tile: stage 5 is reached (whole tiles: no tile's reduction is
    # spread over several pairs, each of which would issue fewer stages)
    H, F, k, M = 1024, 1024, 2, 256
    d = synth.make_inputs(H, F, M, 191)
    dd = inputs_on_device(d)
    Y = torch.empty((M, F), dtype=torch.bfloat16, device="cuda")
    ctx = vp()
    flags = (tp.TPMLP_FLAG_SINGLE_SM if single_sm else 0) | tp.TPMLP_FLAG_FIXED_ORDER
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

