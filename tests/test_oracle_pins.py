"""The fp64 oracle against facts fixed outside it (see tests/oracle_pins.py)."""
import pytest

import oracle
from tests import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check(oracle.default())


def test_bad_rows_rejected():
    import numpy as np
    from io_aware_exact_06_gb300 import inputs
    wl = inputs.make_workload("bad", 1, [4], 1, 4, causal=False)
    with pytest.raises(ValueError):
        oracle.attn_rows(wl.q, wl.k, wl.v, wl.cu_seqlens, np.array([[0, 0, 4]]), 0.5, False)
    with pytest.raises(ValueError):
        oracle.attn_rows(wl.q, wl.k, wl.v, wl.cu_seqlens, np.array([[0, 1, 0]]), 0.5, False)
    with pytest.raises(ValueError):
        oracle.softmax_merge(np.zeros(4), [0])


def test_threads_reported():
    from io_aware_exact_06_gb300 import inputs
    wl = inputs.make_workload("thr", 2, [64], 2, 8, causal=True)
    rows = inputs.all_rows(wl.cu_seqlens, 2)
    o1, l1, used = oracle.attn_rows(wl.q, wl.k, wl.v, wl.cu_seqlens, rows, 0.3, True, 3)
    assert used == 3
    o2, l2, used1 = oracle.attn_rows(wl.q, wl.k, wl.v, wl.cu_seqlens, rows, 0.3, True, 1)
    assert used1 == 1
    assert (o1 == o2).all() and (l1 == l2).all(), "threading changes no result"
