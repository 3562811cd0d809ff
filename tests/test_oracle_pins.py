"""The CPU oracle against its pins (closed forms, a hand-worked example, numpy/scipy routines,
a float64 brute force, the layer's invariants).  CPU only."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(oracle, pin):
    pin(oracle)


def test_oracle_rejects_bad_routing(oracle):
    import numpy as np
    with pytest.raises(ValueError):
        oracle.permute(np.array([[0, 0]], np.int32), 4)      # an expert twice in one token
    with pytest.raises(ValueError):
        oracle.permute(np.array([[0, 4]], np.int32), 4)      # id outside [0, E)
    with pytest.raises(ValueError):
        oracle.route(np.zeros((3, 4), np.float32), 5)        # k > E


def test_oracle_empty_batch(oracle):
    import numpy as np
    idx, w = oracle.route(np.zeros((0, 8), np.float32), 2)
    assert idx.shape == (0, 2) and w.shape == (0, 2)
    counts, offsets, src, dest = oracle.permute(idx, 8)
    assert counts.sum() == 0 and np.all(offsets == 0) and src.size == 0
