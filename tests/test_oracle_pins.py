"""The CPU oracle against what the pages and plain mathematics fix (no GPU needed)."""

import pytest

import oracle
from tests import _pins


@pytest.mark.parametrize("pin", _pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle)


def test_oracle_rejects_bad_inputs():
    import numpy as np
    K = [np.zeros((1, 4, 2), np.float32)]
    pool, pt, sl = _pins.paged_from_contiguous(K, K, 2)
    kv = oracle.PagedKV(pool, pt, sl)
    q = np.zeros((1, 5, 1, 2), np.float32)  # n_c = 5 > L = 4
    with pytest.raises(ValueError):
        oracle.verify(kv, q, 1.0)
    pt_bad = pt.copy()
    pt_bad[0, 1] = 99
    with pytest.raises(ValueError):
        oracle.verify(oracle.PagedKV(pool, pt_bad, sl), np.zeros((1, 1, 1, 2), np.float32), 1.0)
    idx = np.array([[[0, 4]]], np.int32)  # 4 >= L
    with pytest.raises(ValueError):
        oracle.draft(kv, np.zeros((1, 1, 2), np.float32), idx, np.array([[2]], np.int32), 1.0)
