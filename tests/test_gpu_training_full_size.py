"""The training pass at the full 7B shape (X [4, 2048, 4096], F = 16384, k = 8), GeLU and gated,
against the fp64 oracle on samples it can compute exactly:
  - dX on sampled token rows: row m of dX depends only on row m of X and of dZ, so the oracle
    run on those rows alone gives their dX exactly;
  - dW1, db1, dW2 (dWg, dbg, dWu, dbu, dW2 for the gated block) on sampled columns of F: column
    j of the first layer's weight gradient, its bias gradient and row j of dW2 depend only on
    column j of the first layer and row j of W2, so the oracle run on that sub-block (all token
    rows, those columns, k = 1) gives them exactly; its db2 is the whole db2.
The GPU runs the whole problem in one training step."""
import numpy as np
import pytest
import torch

import oracle
import synth
import tensor_transformer_mlp_tmem_gb300 as tp
from gpu_util import assert_close, inputs_on_device, to_dev, to_f64

pytestmark = pytest.mark.gpu


def _sample_cols(F: int, f: int, n: int = 48, seed: int = 7) -> np.ndarray:
    """Columns of F: both edges of every shard boundary, plus a seeded spread."""
    edges = {0, F - 1}
    for i in range(1, F // f):
        edges.update((i * f - 1, i * f))
    rng = np.random.default_rng(seed)
    extra = rng.choice(F, size=n, replace=False)
    return np.array(sorted(edges.union(int(c) for c in extra)), dtype=np.int64)


def _c(a):
    return np.ascontiguousarray(a)


def _check(got: torch.Tensor, ref: np.ndarray, what: str):
    assert_close(to_f64(got).reshape(ref.shape), ref, what=what)


def test_backward_7b_shape_sampled(lib):
    w = synth.WORKLOADS["7b"]
    d = synth.workload_inputs(w)
    dZ = synth.normal_bf16(w.seed, 60, (w.M, w.H), 1.0)
    dd = inputs_on_device(d)
    with tp.TPMLP(w.H, w.F, w.k) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        X = dd["X"].view(w.B, w.S, w.H)
        _, Ys, As = mlp.forward_train(X)
        dX, dW1, db1, dW2, db2 = mlp.backward(to_dev(dZ).view(w.B, w.S, w.H), X, Ys, As,
                                              dd["W1"], dd["W2"])
        torch.cuda.synchronize()
        rc, detail = mlp.status()
        assert rc == tp.TPMLP_OK, f"device status {detail:#x}"
    rows = synth.sample_rows(w.M, 12)
    cols = _sample_cols(w.F, w.F // w.k)
    ref_r = oracle.backward(_c(d["X"][rows]), d["W1"], d["b1"], d["W2"], _c(dZ[rows]), w.k)
    _check(dX.view(w.M, w.H)[torch.from_numpy(rows).cuda()], ref_r["dX"], "dX (sampled rows)")
    ref_c = oracle.backward(d["X"], _c(d["W1"][:, cols]), _c(d["b1"][cols]), _c(d["W2"][cols]), dZ, 1)
    ci = torch.from_numpy(cols).cuda()
    _check(dW1[:, ci], ref_c["dW1"], "dW1 (sampled columns)")
    _check(db1[ci], ref_c["db1"], "db1 (sampled columns)")
    _check(dW2[ci], ref_c["dW2"], "dW2 (sampled rows of W2)")
    _check(db2, ref_c["db2"], "db2")


def test_swiglu_backward_7b_shape_sampled(lib):
    w = synth.WORKLOADS["7b"]
    d = synth.make_swiglu_inputs(w.H, w.F, w.M, w.seed)
    dZ = synth.normal_bf16(w.seed, 60, (w.M, w.H), 1.0)
    dd = inputs_on_device(d)
    with tp.TPMLP(w.H, w.F, w.k, swiglu=True) as mlp:
        mlp.pack_swiglu(dd["Wg"], dd["bg"], dd["Wu"], dd["bu"], dd["W2"], dd["b2"])
        X = dd["X"].view(w.B, w.S, w.H)
        _, Ys, As = mlp.forward_train(X)
        g = mlp.backward_swiglu(to_dev(dZ).view(w.B, w.S, w.H), X, Ys, As, dd["Wg"], dd["Wu"],
                                dd["W2"])
        torch.cuda.synchronize()
        rc, detail = mlp.status()
        assert rc == tp.TPMLP_OK, f"device status {detail:#x}"
    dX, dWg, dbg, dWu, dbu, dW2, db2 = g
    rows = synth.sample_rows(w.M, 12)
    cols = _sample_cols(w.F, w.F // w.k)
    ref_r = oracle.swiglu_backward(_c(d["X"][rows]), d["Wg"], d["bg"], d["Wu"], d["bu"], d["W2"],
                                   _c(dZ[rows]), w.k)
    _check(dX.view(w.M, w.H)[torch.from_numpy(rows).cuda()], ref_r["dX"], "dX (sampled rows)")
    ref_c = oracle.swiglu_backward(d["X"], _c(d["Wg"][:, cols]), _c(d["bg"][cols]),
                                   _c(d["Wu"][:, cols]), _c(d["bu"][cols]), _c(d["W2"][cols]), dZ, 1)
    ci = torch.from_numpy(cols).cuda()
    _check(dWg[:, ci], ref_c["dWg"], "dWg (sampled columns)")
    _check(dbg[ci], ref_c["dbg"], "dbg (sampled columns)")
    _check(dWu[:, ci], ref_c["dWu"], "dWu (sampled columns)")
    _check(dbu[ci], ref_c["dbu"], "dbu (sampled columns)")
    _check(dW2[ci], ref_c["dW2"], "dW2 (sampled rows of W2)")
    _check(db2, ref_c["db2"], "db2")
