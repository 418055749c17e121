"""GPU parity of the block-quantised int8 weight path (weight_dtype SLM_Q8) against the
oracle's Q8 model (kasahare 0.4.0, "Where to go from here": INT8 weights, block-quantised
like GGUF).  Both sides quantise the same fp32 weights (the quantisers agree bit for bit:
tests/test_q8_quantizer.py); the GPU multiplies int8 pieces and applies each block's
scale to the piece's partial sum, the oracle multiplies the dequantised fp32 weights, so
the results differ by rounding only and are held to the usual tolerances (teacher
forcing, gap rule for ids).  Covered: head geometries and ragged widths (partial last
blocks), bf16 and fp32 caches, single rows (8-row groups), batches of 4 and 8, batches of
9..16 rows (the CUDA-core 16-row kernel), K-split residual matrices, and the SmolLM2 shape.
"""
import numpy as np
import pytest

import synth
from parity_util import compare_runs, gpu_teacher_forced, oracle_reference

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

Q8 = synth.DTYPE_Q8


@pytest.fixture(scope="module")
def slm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import llama_decode_kv_gb300 as m
    return m


VARIANTS = {
    "tiny": dict(),
    "mqa_bf16kv": dict(n_kv_heads=1, kv_dtype=synth.DTYPE_BF16),
    "ragged_dims": dict(dim=72, n_heads=3, n_kv_heads=1, head_dim=24, hidden=100, vocab=333),
    "wide_head": dict(dim=256, n_heads=2, n_kv_heads=1, head_dim=128, hidden=300),
    "gqa_hd64_bf16kv": dict(dim=256, n_heads=4, n_kv_heads=1, head_dim=64, hidden=200, kv_dtype=synth.DTYPE_BF16),
}


@pytest.mark.parametrize("name", sorted(VARIANTS))
def test_q8_batched_ragged(slm, name):
    s = synth.TINY.replace(max_batch=3, max_seq=96, weight_dtype=Q8, **VARIANTS[name])
    W = synth.make_weights(s, seed=41)
    assert W.dtype == np.float32
    lens = [3, 9, 40]
    prompts = [synth.make_prompt(s, r, lens[r]) for r in range(3)]
    steps = 6
    ref_ids, ref_logits = oracle_reference(s, prompts, steps, [0, 1, 2], seed=41)
    eng = slm.Engine(s, W)
    assert eng.cluster_plan() is None  # int8 engines run on the persistent kernel
    g_logits, g_ids = gpu_teacher_forced(eng, s, prompts, ref_ids, steps, 3, [0, 1, 2])
    compare_runs(s, ref_ids, ref_logits, g_logits, g_ids, [0, 1, 2], name + " q8")
    eng.close()


@pytest.mark.parametrize("name", ["tiny", "ragged_dims", "gqa_hd64_bf16kv"])
def test_q8_single_row(slm, name):
    s = synth.TINY.replace(max_batch=1, max_seq=64, weight_dtype=Q8, **VARIANTS[name])
    W = synth.make_weights(s, seed=43)
    prompts = [synth.make_prompt(s, 0, 11)]
    steps = 8
    ref_ids, ref_logits = oracle_reference(s, prompts, steps, [0], seed=43)
    eng = slm.Engine(s, W)
    g_logits, g_ids = gpu_teacher_forced(eng, s, prompts, ref_ids, steps, 1, [0])
    compare_runs(s, ref_ids, ref_logits, g_logits, g_ids, [0], name + " q8 single row")
    eng.close()


@pytest.mark.parametrize("batch,hidden", [(8, 200), (13, 200), (16, 200), (12, 2048)])
def test_q8_large_batches(slm, batch, hidden):
    # up to 8 rows: the 8-row kernel; 9..16 rows: the 16-row CUDA-core kernel; hidden
    # 2048 at 16 rows splits W2's input into K tiles (partial sums accumulated)
    s = synth.TINY.replace(max_batch=16, max_seq=96, weight_dtype=Q8, kv_dtype=synth.DTYPE_BF16, dim=128,
                           n_heads=4, n_kv_heads=2, head_dim=32, hidden=hidden, vocab=300)
    W = synth.make_weights(s, seed=47)
    lens = [3 + (7 * r) % 40 for r in range(batch)]
    prompts = [synth.make_prompt(s, r, lens[r]) for r in range(batch)]
    steps = 3
    rows = list(range(batch))
    ref_ids, ref_logits = oracle_reference(s, prompts, steps, rows, seed=47)
    eng = slm.Engine(s, W)
    g_logits, g_ids = gpu_teacher_forced(eng, s, prompts, ref_ids, steps, batch, rows)
    compare_runs(s, ref_ids, ref_logits, g_logits, g_ids, rows, f"q8 batch {batch} hidden {hidden}")
    eng.close()


def test_q8_smol_shape(slm):
    """The SmolLM2-135M shape with int8 weights (151 MB on the device instead of 269 MB of
    bf16), batch 1, fp32 cache: every logit of 8 steps against the oracle."""
    s = synth.SMOL.replace(weight_dtype=Q8, max_seq=64)
    W = synth.make_weights(s, seed=53)
    prompts = [synth.make_prompt(s, 0, 5)]
    steps = 8
    ref_ids, ref_logits = oracle_reference(s, prompts, steps, [0], seed=53)
    eng = slm.Engine(s, W)
    g_logits, g_ids = gpu_teacher_forced(eng, s, prompts, ref_ids, steps, 1, [0])
    compare_runs(s, ref_ids, ref_logits, g_logits, g_ids, [0], "smol q8")
    eng.close()
