"""Cache replication (slm_fork) on the GPU.

"Inside nanochat Part 4: Understanding Inference", Batch Prefilling via Cache
Replication: one prompt is prefilled at batch 1 and its cache is copied to N rows that
then generate independently.  The clone must be byte-exact, and every row continued from
it must decode exactly as if it had been prefilled on its own (checked against the
oracle, which prefills each row independently).
"""
import numpy as np
import pytest
import torch

import synth
from parity_util import compare_runs, oracle_reference

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def slm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import llama_decode_kv_gb300 as m
    return m


@pytest.mark.parametrize("kv", [synth.DTYPE_F32, synth.DTYPE_BF16])
def test_fork_copies_the_cache_byte_for_byte(slm, kv):
    s = synth.TINY.replace(max_batch=5, max_seq=48, weight_dtype=synth.DTYPE_BF16, kv_dtype=kv)
    eng = slm.Engine(s, synth.make_weights(s, seed=5))
    prompt = synth.make_prompt(s, 0, 21)
    eng.prefill_checked(2, prompt, want_logits=False)
    assert eng.fork(2, [4, 0, 1]) == 0, eng.last_error()
    assert eng.sync() == 0
    for d in (4, 0, 1):
        assert eng.seq_len(d) == 21
    assert eng.seq_len(3) == 0
    for layer in range(s.n_layers):
        k_src, v_src = eng.kv(layer, 2)
        for d in (4, 0, 1):
            k, v = eng.kv(layer, d)
            assert np.array_equal(k.view(np.uint32), k_src.view(np.uint32)), (layer, d)
            assert np.array_equal(v.view(np.uint32), v_src.view(np.uint32)), (layer, d)
    eng.close()


@pytest.mark.parametrize("kv", [synth.DTYPE_F32, synth.DTYPE_BF16])
def test_rows_continued_from_a_fork_match_independent_prefills(slm, kv):
    # prompt P prefilled once on row 0 and cloned to rows 1..3; row r then decodes its own
    # token t_r at position len(P) and continues.  The oracle prefills P + [t_r] per row.
    s = synth.TINY.replace(max_batch=4, max_seq=64, weight_dtype=synth.DTYPE_BF16, kv_dtype=kv)
    W = synth.make_weights(s, seed=7)
    P = synth.make_prompt(s, 0, 18)
    tails = [3, 77, 150, 201]
    rows = list(range(4))
    prompts = [np.concatenate([P, np.array([t], dtype=np.int32)]) for t in tails]
    steps = 5
    ref_ids, ref_logits = oracle_reference(s, prompts, steps, rows, seed=7)

    eng = slm.Engine(s, W)
    dev = torch.device("cuda")
    eng.prefill_checked(0, P, want_logits=False)
    assert eng.fork(0, [1, 2, 3]) == 0, eng.last_error()
    g_logits = {r: [] for r in rows}
    g_ids = {r: [] for r in rows}
    cur = list(tails)
    for st in range(steps + 1):
        toks = torch.tensor(cur, dtype=torch.int32, device=dev)
        lg, nid = eng.decode_checked(rows, toks, [len(P) + st] * 4, want_logits=True)
        lg, nid = lg.cpu().numpy(), nid.cpu().numpy()
        for r in rows:
            g_logits[r].append(lg[r])
            g_ids[r].append(int(nid[r]))
            if st < steps:
                cur[r] = ref_ids[r][st]  # teacher forcing with the oracle's ids
    assert eng.sync() == 0, eng.last_error()
    compare_runs(s, ref_ids, ref_logits, g_logits, g_ids, rows, f"fork kv={kv}")
    eng.close()


def test_fork_refuses_bad_arguments_and_changes_nothing(slm):
    s = synth.TINY.replace(max_batch=4, max_seq=32)
    eng = slm.Engine(s, synth.make_weights(s))
    EINVAL, ESTATE = -1, -5
    assert eng.fork(0, [1]) == ESTATE  # empty source
    eng.prefill_checked(0, synth.make_prompt(s, 0, 6), want_logits=False)
    eng.prefill_checked(3, synth.make_prompt(s, 3, 4), want_logits=False)
    assert eng.fork(0, [3]) == ESTATE  # destination not empty
    assert eng.fork(0, [1, 3]) == ESTATE
    assert eng.fork(0, [0]) == EINVAL  # destination is the source
    assert eng.fork(0, [1, 1]) == EINVAL  # repeated
    assert eng.fork(0, [4]) == EINVAL  # out of range
    assert eng.fork(-1, [1]) == EINVAL
    assert eng.fork(0, []) == EINVAL
    assert [eng.seq_len(q) for q in range(4)] == [6, 0, 0, 4]
    assert eng.fork(0, [1, 2]) == 0
    assert eng.sync() == 0
    assert [eng.seq_len(q) for q in range(4)] == [6, 6, 6, 4]
    eng.close()
