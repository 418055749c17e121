"""Pins of the oracle's block-quantised int8 weights (orc_quantize_q8_row, weight dtype
Q8), each against something outside the oracle: exact integer grids, the rounding rule
written out by hand, the textbook round-to-nearest error bound, and the fp64 model walk.

Format (kasahare 0.4.0, "Where to go from here": INT8 weights, block-quantised like
GGUF; the pages give no layout, so the plainest one): blocks of 32 consecutive elements
of a row, d = max|w| / 127, q = round(w / d) with halves away from zero, weight = d * q.
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def test_exact_grid_is_reproduced():
    # w = k * 2^-7 with integers |k| <= 127 and one |k| = 127 per block: d = 2^-7
    # exactly (127 * 2^-7 / 127 is exact), so q = k and d * q = w bit for bit
    rng = np.random.default_rng(3)
    k = rng.integers(-127, 128, 96).astype(np.int32)
    k[5], k[40], k[70] = 127, -127, 127
    w = (k * 2.0 ** -7).astype(np.float32)
    q, d = oracle.quantize_q8_row(w)
    assert np.array_equal(q.astype(np.int32), k)
    assert np.array_equal(d, np.full(3, 2.0 ** -7, dtype=np.float32))
    assert np.array_equal(d[np.arange(96) // 32] * q.astype(np.float32), w)


def test_halves_round_away_from_zero():
    # a block with max|w| = 127 has d = 1, so q is w rounded to an integer
    w = np.zeros(32, dtype=np.float32)
    w[:8] = [127.0, 2.5, -2.5, 0.5, -0.5, 1.49, -1.51, 126.5]
    q, d = oracle.quantize_q8_row(w)
    assert d[0] == 1.0
    assert list(q[:8]) == [127, 3, -3, 1, -1, 1, -2, 127]


def test_zero_block_and_partial_last_block():
    # 72 elements = blocks of 32, 32 and 8; the middle block is all zero; the last
    # block's scale comes from its own 8 elements only
    w = np.zeros(72, dtype=np.float32)
    w[:32] = np.linspace(-1.0, 1.0, 32, dtype=np.float32)
    w[64:] = np.array([0.0, 0.25, -0.5, 0.125, 0.0, 0.0, 0.375, -0.0625], dtype=np.float32)
    q, d = oracle.quantize_q8_row(w)
    assert d.shape == (3,)
    assert d[1] == 0.0 and not np.any(q[32:64])
    assert d[2] == np.float32(0.5) / np.float32(127.0)
    assert q[66] == -127
    assert d[0] == np.float32(1.0) / np.float32(127.0) and q[0] == -127 and q[31] == 127


def test_error_bound_and_full_scale():
    # round to nearest: |w - d q| <= d / 2 (plus the rounding of w / d and of d q); the
    # largest element of every nonzero block maps to +-127
    rng = np.random.default_rng(11)
    w = (rng.standard_normal(32 * 50) * 0.02).astype(np.float32)
    q, d = oracle.quantize_q8_row(w)
    blk = np.arange(w.size) // 32
    deq = d[blk].astype(np.float64) * q.astype(np.float64)
    err = np.abs(w.astype(np.float64) - deq)
    assert np.all(err <= d[blk].astype(np.float64) * (0.5 + 1e-5))
    for b in range(50):
        seg = w[32 * b:32 * (b + 1)]
        i = int(np.argmax(np.abs(seg)))
        assert abs(int(q[32 * b + i])) == 127
        assert np.all(np.abs(q[32 * b:32 * (b + 1)].astype(np.int32)) <= 127)


def test_q8_model_is_the_model_of_the_dequantised_weights():
    # every matrix (embedding, q, k, v, o, w1, w3, w2) is quantised row by row and the
    # norms are not: the Q8 oracle's logits equal the fp64 decoder run on weights that
    # this test dequantises itself from the pinned row quantiser
    s = synth.TINY.replace(weight_dtype=synth.DTYPE_Q8, dim=72, n_heads=3, n_kv_heads=1, head_dim=24, hidden=100,
                           vocab=333, max_seq=16)
    W = synth.make_weights(s, seed=7)
    assert W.dtype == np.float32
    W = W.copy()
    for name, _layer, off, count in synth.layout(s):  # every block visibly moves the residual
        if not name.endswith("norm") and name != "token_emb":
            W[off:off + count] *= 10
    Wq = W.copy()
    for name, _layer, off, count in synth.layout(s):
        if name.endswith("norm"):
            continue
        n_in = s.hidden if name == "w2" else (s.n_heads * s.head_dim if name == "wo" else s.dim)
        rows = Wq[off:off + count].reshape(-1, n_in)
        for r in range(rows.shape[0]):
            q, d = oracle.quantize_q8_row(rows[r])
            rows[r] = d[np.arange(n_in) // 32] * q.astype(np.float32)
    tokens = synth.make_prompt(s, 0, 6)
    o = oracle.Model(s, W)
    lg, _ = o.prefill(0, tokens)
    from test_oracle_pins import _decoder_fp64
    ref = _decoder_fp64(s.replace(weight_dtype=synth.DTYPE_F32), Wq, tokens)
    assert np.max(np.abs(lg - ref)) <= 1e-5 * np.max(np.abs(ref))
    # and the quantisation matters: the unquantised weights give visibly different logits
    lg32, _ = oracle.Model(s.replace(weight_dtype=synth.DTYPE_F32), W).prefill(0, tokens)
    assert np.max(np.abs(lg32 - lg)) > 1e-3 * np.max(np.abs(ref))
