"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle on the same
seeded inputs, on every workload shape, ragged token counts and the degenerate cases."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
import tensor_transformer_mlp_tmem_gb300 as tp
from gpu_util import (K_INVARIANCE_BAR, assert_close, bits_of, device_tensor, f64,
                      inputs_on_device, max_abs_rel, rel_fro, to_dev, to_f64)

pytestmark = pytest.mark.gpu


def run_block(d, H, F, k, M, z_fp32=False):
    dd = inputs_on_device(d)
    with tp.TPMLP(H, F, k, z_fp32=z_fp32) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        Z = mlp(dd["X"].view(1, M, H))
        rc, detail = mlp.status()
        assert rc == tp.TPMLP_OK, f"device status {detail:#x}"
    return to_f64(Z.view(M, H))


# ----------------------------------------------------------------------------- packer
@pytest.mark.parametrize("H,F,k", [(256, 1024, 2), (512, 2048, 4), (128, 512, 4), (64, 256, 4)])
def test_pack_layout_is_exact_permutation(lib, H, F, k):
    d = synth.make_inputs(H, F, 4, 21)
    dd = inputs_on_device(d)
    f = F // k
    with tp.TPMLP(H, F, k) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        torch.cuda.synchronize()
        p, n = tp.tpmlp_packed_buffer(mlp.ctx, 0)
        assert n == H * F * 2
        W1p = device_tensor(p, (k, f, H), "i16").cpu().numpy().view(np.uint16)
        p, _ = tp.tpmlp_packed_buffer(mlp.ctx, 1)
        if H % 256 == 0:
            # second GEMM on CTA pairs: 16 KB blocks [k][H/128][f/64][128][64]
            W2b = device_tensor(p, (k, H // 128, f // 64, 128, 64), "i16").cpu().numpy()
            W2p = W2b.transpose(0, 1, 3, 2, 4).reshape(k, H, f).view(np.uint16)
        else:
            W2p = device_tensor(p, (k, H, f), "i16").cpu().numpy().view(np.uint16)
        p, _ = tp.tpmlp_packed_buffer(mlp.ctx, 2)
        b1p = device_tensor(p, (F,), "f32").cpu().numpy()
        p, _ = tp.tpmlp_packed_buffer(mlp.ctx, 3)
        b2p = device_tensor(p, (H,), "f32").cpu().numpy()
    for i in range(k):
        # column shard i of W1, transposed; row shard i of W2, transposed
        assert np.array_equal(W1p[i], d["W1"][:, i * f:(i + 1) * f].T)
        assert np.array_equal(W2p[i], d["W2"][i * f:(i + 1) * f, :].T)
    assert np.array_equal(b1p.astype(np.float64), f64(d["b1"]))
    assert np.array_equal(b2p.astype(np.float64), f64(d["b2"]))


# ----------------------------------------------------------------------------- GEMM1 alone
@pytest.mark.parametrize("H,F,k,M", [(256, 1024, 2, 128), (128, 512, 4, 300), (64, 256, 4, 77)])
def test_gemm1_matches_oracle_activations(lib, H, F, k, M):
    d = synth.make_inputs(H, F, M, 5)
    dd = inputs_on_device(d)
    with tp.TPMLP(H, F, k) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        Y = mlp.gemm1(dd["X"])
        torch.cuda.synchronize()
    ref = oracle.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], k, want_y=True)["Y"]
    assert_close(to_f64(Y), ref, what="Y (concatenated shard activations)")


# ----------------------------------------------------------------------------- workloads
@pytest.mark.parametrize("name,rows", [("tiny", None), ("gpt2-small", None), ("7b", 64),
                                       ("gpt3-175b", 24)])
def test_forward_matches_oracle_on_workload(lib, name, rows):
    w = synth.WORKLOADS[name]
    d = synth.workload_inputs(w)
    z = run_block(d, w.H, w.F, w.k, w.M)
    sel = None if rows is None else synth.sample_rows(w.M, rows)
    ref = oracle.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], w.k, rows=sel)["Z"]
    got = z if sel is None else z[sel]
    r, m = assert_close(got, ref, what=name)
    print(f"{name}: rel_fro={r:.3e} max_abs/max|Z|={m:.3e}")
    assert np.all(np.isfinite(z))


def test_token_count_past_32_bit_element_offsets(lib):
    """The 7B-shaped block at M = 135168 tokens (B = 33, S = 4096): Y [M, F] holds 2.2e9
    elements, past 2^31, so the last row blocks' Y and Z addresses need 64-bit index math in
    both kernels' epilogue stores and in the tensor maps the second GEMM reads Y through. Rows
    on both sides of the 2^31-element boundary of Y, the last row and a seeded spread are
    checked against the oracle."""
    w = synth.WORKLOADS["7b"]
    B, S = 33, 4096
    M = B * S
    edge = (1 << 31) // w.F  # first row of Y whose elements start at or past 2^31
    assert (M - 1) * w.F >= 1 << 31 and edge < M
    d = synth.make_inputs(w.H, w.F, M, 17)
    sel = np.array(sorted(set(synth.sample_rows(M, 24).tolist()) |
                          {edge - 1, edge, edge + 1, M - 1}), dtype=np.int64)
    dd = inputs_on_device(d)
    with tp.TPMLP(w.H, w.F, w.k) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        Z = mlp(dd["X"].view(B, S, w.H))
        torch.cuda.synchronize()
        rc, detail = mlp.status()
        assert rc == tp.TPMLP_OK, f"device status {detail:#x}"
        z = to_f64(Z.view(M, w.H)[torch.from_numpy(sel).cuda()])
    ref = oracle.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], w.k, rows=sel)["Z"]
    assert np.all(np.isfinite(z))
    assert_close(z, ref, what=f"7b shape, M = {M}")


def test_shard_count_sweep(lib):
    """Sweep workload: identical inputs for k = 1, 2, 4, 8, 16; each k against the oracle
    on sampled rows, and every k against k = 1 over the whole output."""
    w = synth.WORKLOADS["sweep-h4096"]
    d = synth.workload_inputs(w)
    sel = synth.sample_rows(w.M, 24)
    outs = {}
    for k in w.ks:
        z = run_block(d, w.H, w.F, k, w.M)
        ref = oracle.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], k, rows=sel)["Z"]
        assert_close(z[sel], ref, what=f"sweep k={k}")
        outs[k] = z
    for k in w.ks:
        r = rel_fro(outs[k], outs[1])
        assert r <= K_INVARIANCE_BAR, f"k={k} vs k=1: rel_fro={r:.3e}"
    print("sweep k=8 vs k=1 rel_fro:", rel_fro(outs[8], outs[1]))


# ----------------------------------------------------------------------------- edges
@pytest.mark.parametrize("M", [1, 5, 127, 129, 255, 300, 1000])
def test_ragged_token_counts(lib, M):
    H, F, k = 256, 1024, 4
    d = synth.make_inputs(H, F, M, 31)
    z = run_block(d, H, F, k, M)
    ref = oracle.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], k)["Z"]
    assert_close(z, ref, what=f"M={M}")


@pytest.mark.parametrize("H,F,k", [
    (64, 256, 4),      # narrowest shard (f = 64) and narrowest output tile
    (64, 4096, 64),    # maximum shard count for F (f = 64)
    (384, 1536, 2),    # 128-wide output tiles in the second GEMM
    (320, 1280, 5),    # 64-wide tiles in both GEMMs, odd k
    (768, 3072, 1),    # unsharded
])
def test_tile_widths_and_shard_counts(lib, H, F, k):
    M = 200
    d = synth.make_inputs(H, F, M, 41)
    z = run_block(d, H, F, k, M)
    ref = oracle.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], k)["Z"]
    assert_close(z, ref, what=f"H={H} F={F} k={k}")


def test_fp32_output(lib):
    H, F, k, M = 256, 1024, 2, 256
    d = synth.make_inputs(H, F, M, 51)
    z = run_block(d, H, F, k, M, z_fp32=True)
    ref = oracle.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], k)["Z"]
    r, m = assert_close(z, ref, rel=5e-3, mx=2e-2, what="fp32 Z")


def test_empty_batch_is_noop(lib):
    H, F, k = 256, 1024, 2
    d = synth.make_inputs(H, F, 1, 3)
    dd = inputs_on_device(d)
    with tp.TPMLP(H, F, k) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        n0 = mlp.launches
        X = torch.empty((0, 64, H), dtype=torch.bfloat16, device="cuda")
        Z = mlp(X)
        assert Z.shape == (0, 64, H) and mlp.launches == n0


def test_staged_calls_equal_forward_and_are_deterministic(lib):
    H, F, k, M = 256, 1024, 4, 384
    d = synth.make_inputs(H, F, M, 61)
    dd = inputs_on_device(d)
    with tp.TPMLP(H, F, k) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        Z1 = mlp(dd["X"].view(1, M, H))
        Z2 = mlp(dd["X"].view(1, M, H))
        Y = mlp.gemm1(dd["X"])
        Z3 = mlp.gemm2(Y)
        torch.cuda.synchronize()
    assert torch.equal(Z1, Z2)
    assert torch.equal(Z1.view(M, H), Z3)


def test_forward_host_equals_device(lib):
    H, F, k, M = 256, 1024, 2, 256
    d = synth.make_inputs(H, F, M, 71)
    dd = inputs_on_device(d)
    Xh = torch.from_numpy(d["X"].view(np.int16)).view(torch.bfloat16).pin_memory()
    Zh = torch.empty((M, H), dtype=torch.bfloat16).pin_memory()
    with tp.TPMLP(H, F, k) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        Zd = mlp(dd["X"].view(1, M, H))
        torch.cuda.synchronize()
        tp.tpmlp_forward_host(mlp.ctx, Xh, 1, M, Zh)
    assert torch.equal(Zd.view(M, H).cpu(), Zh)


def test_guard_bands_untouched(lib):
    """Canary words around the caller's Y and Z buffers stay intact (stands in for a
    memory checker: every store of both kernels lands inside its output)."""
    H, F, k, M = 256, 1024, 2, 200
    d = synth.make_inputs(H, F, M, 81)
    dd = inputs_on_device(d)
    G = 4096  # guard elements on each side (multiple of 8: keeps 16-byte alignment)
    sentinel = -12345
    ybuf = torch.full((G + M * F + G,), sentinel, dtype=torch.int16, device="cuda")
    zbuf = torch.full((G + M * H + G,), sentinel, dtype=torch.int16, device="cuda")
    Y = ybuf[G:G + M * F].view(torch.bfloat16).view(M, F)
    Z = zbuf[G:G + M * H].view(torch.bfloat16).view(M, H)
    with tp.TPMLP(H, F, k) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        mlp.gemm1(dd["X"], Y)
        mlp.gemm2(Y, Z)
        torch.cuda.synchronize()
    for buf, n in ((ybuf, M * F), (zbuf, M * H)):
        assert torch.all(buf[:G] == sentinel) and torch.all(buf[G + n:] == sentinel)
    ref = oracle.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], k)["Z"]
    assert_close(to_f64(Z), ref, what="guarded Z")


def test_argument_errors_on_device(lib):
    H, F, k = 256, 1024, 2
    d = synth.make_inputs(H, F, 128, 3)
    dd = inputs_on_device(d)
    Z = torch.empty((128, H), dtype=torch.bfloat16, device="cuda")
    with tp.TPMLP(H, F, k) as mlp:
        with pytest.raises(tp.TpmlpError) as e:
            tp.tpmlp_forward(mlp.ctx, dd["X"], 1, 128, Z)
        assert e.value.status == tp.TPMLP_ERR_NOT_PACKED
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        with pytest.raises(tp.TpmlpError) as e:
            tp.tpmlp_forward(mlp.ctx, dd["X"].data_ptr() + 2, 1, 127, Z)
        assert e.value.status == tp.TPMLP_ERR_MISALIGNED
        with pytest.raises(tp.TpmlpError) as e:
            tp.tpmlp_forward(mlp.ctx, dd["X"], -1, 128, Z)
        assert e.value.status == tp.TPMLP_ERR_INVALID_ARG
        assert mlp.status()[0] == tp.TPMLP_OK


# ----------------------------------------------------------------------------- both kernels
@pytest.mark.parametrize("H,F,k,M", [(256, 1024, 2, 128), (256, 1024, 4, 777), (1024, 4096, 4, 1000),
                                     (512, 2048, 8, 4096), (768, 3072, 3, 300)])
def test_pair_and_single_sm_kernels_agree(lib, H, F, k, M):
    """With TPMLP_FLAG_FIXED_ORDER the CTA-pair kernel (256 x 256 tiles on two SMs) and the
    single-SM kernel (128-row tiles) reduce in the same order, so Y and Z agree bit for bit;
    the default schedule (which may split the last tiles' reductions) matches the oracle."""
    d = synth.make_inputs(H, F, M, 101)
    dd = inputs_on_device(d)
    outs = []
    for single, fixed in ((True, True), (False, True), (False, False)):
        with tp.TPMLP(H, F, k, single_sm=single, fixed_order=fixed) as mlp:
            mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
            Y = mlp.gemm1(dd["X"])
            Z = mlp.gemm2(Y)
            torch.cuda.synchronize()
            assert mlp.status()[0] == tp.TPMLP_OK
            outs.append((bits_of(Y), bits_of(Z)))
    assert np.array_equal(outs[0][0], outs[1][0]), "Y differs between kernels"
    assert np.array_equal(outs[0][1], outs[1][1]), "Z differs between kernels"
    ref = oracle.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], k)["Z"]
    assert_close(f64(outs[1][1]), ref, what=f"pair kernel H={H} F={F} k={k} M={M}")
    assert_close(f64(outs[2][1]), ref, what=f"pair kernel, default schedule, H={H} F={F} k={k} M={M}")


def test_single_sm_kernel_on_a_large_workload(lib):
    """7B-shaped block with the single-SM kernel forced (sampled rows vs the oracle)."""
    w = synth.WORKLOADS["7b"]
    d = synth.workload_inputs(w)
    dd = inputs_on_device(d)
    with tp.TPMLP(w.H, w.F, w.k, single_sm=True) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        Z = mlp(dd["X"].view(w.B, w.S, w.H))
        torch.cuda.synchronize()
        assert mlp.status()[0] == tp.TPMLP_OK
    sel = synth.sample_rows(w.M, 32)
    ref = oracle.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], w.k, rows=sel)["Z"]
    assert_close(to_f64(Z.view(w.M, w.H))[sel], ref, what="7b single-SM")


@pytest.mark.parametrize("pinned_z", [True, False], ids=["Z-pinned", "Z-pageable"])
@pytest.mark.parametrize("M", [4096, 8192 + 300])
def test_forward_host_pipelined_chunks(lib, M, pinned_z):
    """Large token counts go through the planned chunks of the copy/compute pipeline (copies
    in and out on the context's copy streams, page-locked or pageable host memory). With
    TPMLP_FLAG_FIXED_ORDER the result equals the device-buffer forward bit for bit; by default
    the chunks' split plans may differ from the whole batch's, so the two agree up to fp32
    summation order."""
    H, F, k = 512, 2048, 4
    d = synth.make_inputs(H, F, M, 201)
    dd = inputs_on_device(d)
    Xh = torch.from_numpy(d["X"].view(np.int16)).view(torch.bfloat16).pin_memory()
    for fixed in (True, False):
        Zh = torch.full((M, H), float("nan"), dtype=torch.bfloat16)
        if pinned_z:
            Zh = Zh.pin_memory()
        with tp.TPMLP(H, F, k, fixed_order=fixed) as mlp:
            mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
            Zd = mlp(dd["X"].view(1, M, H))
            torch.cuda.synchronize()
            tp.tpmlp_forward_host(mlp.ctx, Xh, 1, M, Zh)
            tp.tpmlp_forward_host(mlp.ctx, Xh, 1, M, Zh)  # twice: staging and events reused
            assert mlp.status()[0] == tp.TPMLP_OK
        if fixed:
            assert torch.equal(Zd.view(M, H).cpu(), Zh)
        else:
            assert_close(to_f64(Zh), to_f64(Zd.view(M, H).cpu()), rel=2e-3, mx=1e-2,
                         what="host-buffer forward vs device forward")
