"""The CPU oracle against its pins (no GPU)."""
import numpy as np
import pytest

import oracle
import synth
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oracle.default())


def test_oracle_rejects_bad_shard_count():
    d = synth.make_inputs(64, 256, 4, 0)
    with pytest.raises(ValueError):
        oracle.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], 3)  # 256 % 3 != 0


def test_oracle_rejects_row_out_of_range():
    d = synth.make_inputs(64, 256, 4, 0)
    with pytest.raises(ValueError):
        oracle.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], 2, rows=[0, 4])


def test_oracle_empty_rows():
    d = synth.make_inputs(64, 256, 4, 0)
    r = oracle.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], 2, rows=np.zeros(0, np.int64))
    assert r["Z"].shape == (0, 64)
