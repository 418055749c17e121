"""The library's int8 block quantiser (slm_quantize_q8, a host function: no GPU) gives
the same int8 values and scales as the oracle's, bit for bit, on random rows of every
width class (one block, partial blocks, many blocks) and on the special cases (zero
blocks, exact grids, halves).  Integer work: compared exactly."""
import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module")
def slm():
    import llama_decode_kv_gb300 as m
    return m


@pytest.mark.parametrize("cols", [1, 7, 31, 32, 33, 72, 100, 576, 2048])
def test_random_rows_match_oracle(slm, cols):
    rng = np.random.default_rng(cols)
    w = (rng.standard_normal((9, cols)) * np.exp(rng.uniform(-8, 2, (9, 1)))).astype(np.float32)
    w[3] = 0.0                       # an all-zero row
    w[4, : min(cols, 40)] = 0.0      # zero blocks next to nonzero ones
    q, d = slm.quantize_q8(w)
    for r in range(w.shape[0]):
        oq, od = oracle.quantize_q8_row(w[r])
        assert np.array_equal(q[r], oq), f"row {r}"
        assert np.array_equal(d[r].view(np.uint32), od.view(np.uint32)), f"row {r}"


def test_special_values_match_oracle(slm):
    w = np.zeros((3, 64), dtype=np.float32)
    w[0, :8] = [127.0, 2.5, -2.5, 0.5, -0.5, 1.49, -1.51, 126.5]   # d = 1: rounding of halves
    w[1] = (np.arange(64) - 32) * 2.0 ** -7                          # an exact grid
    w[2, 1] = -3e-30                                                 # tiny scales
    q, d = slm.quantize_q8(w)
    for r in range(3):
        oq, od = oracle.quantize_q8_row(w[r])
        assert np.array_equal(q[r], oq) and np.array_equal(d[r], od)
    assert list(q[0, :8]) == [127, 3, -3, 1, -1, 1, -2, 127]


def test_bad_arguments(slm):
    assert slm.slm_quantize_q8(None, 1, 4, None, None) == slm.SLM_EINVAL
