"""GPU tests of the paged KV cache (slm_config.kv_page_size > 0).

Results must not depend on the cache layout ("Inside nanochat Part 4: Understanding
Inference", Continuous Batching: sequences join and leave a running batch, so their
cache lives in pages taken from a shared pool): every test runs the same inputs through
a contiguous engine and a paged one whose pages are scattered on purpose (a scratch
sequence takes pages first and returns them, so the rows' later pages come back in
reverse order), and asks for bit-identical logits and ids; the paged run is also compared
with the oracle (teacher forcing).  Covered: the batched decode kernel (whole-chunk copies
and streamed chunks), the single-row cluster kernel, the tensor-core prefill, slm_fork's
shared pages and copy on write, and pool exhaustion.
"""
import numpy as np
import pytest

import synth
from parity_util import check_logits, compare_runs, oracle_reference, tolerance

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def slm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import llama_decode_kv_gb300 as m
    return m


def _run(slm, s, W, prompts, ref_ids, steps, page, rows=(0, 1, 2), scatter=True, single=False, pages=0):
    """Prefill `rows` (after a scratch sequence took and returned pages, when scatter),
    then `steps` teacher-forced decode steps (batched, or one row at a time with single).
    Returns (logits[r][step], ids[r][step], engine)."""
    eng = slm.Engine(s, W, kv_page_size=page, kv_pages=pages)
    dev = torch.device("cuda")
    scratch = s.max_batch - 1
    if scatter:
        eng.prefill_checked(scratch, synth.make_prompt(s, 99, 45), want_logits=False)
    logits = {r: [] for r in rows}
    ids = {r: [] for r in rows}
    for r in rows:
        lg, nid = eng.prefill_checked(r, prompts[r], want_logits=True)
        logits[r].append(lg.cpu().numpy())
        ids[r].append(int(nid.item()))
    if scatter:
        eng.reset(scratch)
    for st in range(steps):
        groups = [[r] for r in rows] if single else [list(rows)]
        for grp in groups:
            tok = torch.tensor([ref_ids[r][st] for r in grp], dtype=torch.int32, device=dev)
            lg, nid = eng.decode_checked(grp, tok, [len(prompts[r]) + st for r in grp], want_logits=True)
            lg = lg.cpu().numpy()
            nid = nid.cpu().numpy()
            for i, r in enumerate(grp):
                logits[r].append(lg[i])
                ids[r].append(int(nid[i]))
    assert eng.sync() == 0, eng.last_error()
    return logits, ids, eng


def _same(a, b, rows, what):
    for r in rows:
        for st, (x, y) in enumerate(zip(a[r], b[r])):
            assert np.array_equal(x, y), f"{what}: row {r} step {st} differs from the contiguous cache"


PAGED_SHAPES = {
    "fp32kv_hd16": dict(),
    "bf16kv_hd64_g4": dict(kv_dtype=synth.DTYPE_BF16, dim=256, n_heads=4, n_kv_heads=1, head_dim=64),
    "fp32kv_hd128": dict(dim=256, n_heads=2, n_kv_heads=1, head_dim=128, hidden=300),
}


@pytest.mark.parametrize("streamed", [False, True])
@pytest.mark.parametrize("name", sorted(PAGED_SHAPES))
def test_paged_batched_decode(slm, name, streamed, monkeypatch):
    if streamed:  # long chunks read through the per-warp rings, across page boundaries
        monkeypatch.setenv("SLM_ATTN_CHUNK", "64")
        monkeypatch.setenv("SLM_ATTN_STAGE", "0")
    s = synth.TINY.replace(max_batch=4, max_seq=256, **PAGED_SHAPES[name])
    W = synth.make_weights(s, seed=23)
    lens = [21, 70, 133]  # mid-page ends; several pages each
    prompts = [synth.make_prompt(s, r, lens[r]) for r in range(3)]
    steps = 12  # rows cross page boundaries while decoding
    ref_ids, ref_logits = oracle_reference(s, prompts, steps, [0, 1, 2], seed=23)
    c_log, c_ids, ce = _run(slm, s, W, prompts, ref_ids, steps, page=0, scatter=False)
    ce.close()
    p_log, p_ids, pe = _run(slm, s, W, prompts, ref_ids, steps, page=16)
    tables = [pe.page_table(r) for r in range(3)]
    assert any(np.any(np.diff(t[t >= 0]) != 1) for t in tables), "pages should be scattered"
    pe.close()
    _same(c_log, p_log, [0, 1, 2], name)
    assert c_ids == p_ids
    compare_runs(s, ref_ids, ref_logits, p_log, p_ids, [0, 1, 2], name + " paged")


def test_paged_single_row_and_tensor_core_prefill(slm):
    """Single-row steps (the cluster kernel) and prompts long enough for the tensor-core
    prefill, on 32-position pages."""
    s = synth.TINY.replace(max_batch=3, max_seq=160, kv_dtype=synth.DTYPE_BF16, dim=256, n_heads=4, n_kv_heads=1,
                           head_dim=64)
    W = synth.make_weights(s, seed=29)
    lens = [40, 97]
    prompts = [synth.make_prompt(s, r, lens[r]) for r in range(2)]
    steps = 6
    ref_ids, ref_logits = oracle_reference(s, prompts, steps, [0, 1], seed=29)
    c_log, c_ids, ce = _run(slm, s, W, prompts, ref_ids, steps, page=0, rows=(0, 1), scatter=False, single=True)
    assert ce.cluster_plan() is not None
    ce.close()
    p_log, p_ids, pe = _run(slm, s, W, prompts, ref_ids, steps, page=32, rows=(0, 1), single=True)
    pe.close()
    _same(c_log, p_log, [0, 1], "single rows")
    assert c_ids == p_ids
    compare_runs(s, ref_ids, ref_logits, p_log, p_ids, [0, 1], "single rows paged")


def test_paged_fork_shares_pages_and_copies_on_write(slm):
    """slm_fork on a paged cache takes no page; the clones' first steps each copy the
    shared partial page (the source's last page stays with whoever writes last); every
    clone then decodes its own continuation exactly as on a contiguous cache, where the
    fork copies bytes."""
    s = synth.TINY.replace(max_batch=4, max_seq=128, kv_dtype=synth.DTYPE_BF16, dim=256, n_heads=4, n_kv_heads=1,
                           head_dim=64)
    W = synth.make_weights(s, seed=31)
    prompt = synth.make_prompt(s, 0, 37)  # 37 = 2 full pages of 16 + 5
    dev = torch.device("cuda")
    outs = {}
    for page in (0, 16):
        eng = slm.Engine(s, W, kv_page_size=page)
        _, nid = eng.prefill_checked(0, prompt, want_logits=False)
        free0 = eng.pages_free()
        assert eng.fork(0, [1, 2, 3]) == 0, eng.last_error()
        if page:
            assert eng.pages_free() == free0
            t0 = eng.page_table(0)
            for r in (1, 2, 3):
                assert np.array_equal(eng.page_table(r)[:3], t0[:3])
        # each row continues with its own tokens (row r feeds (first id + 7 r) mod vocab)
        toks = [(int(nid.item()) + 7 * r) % s.vocab for r in range(4)]
        res = []
        fed = []
        for st in range(20):
            fed.append(list(toks))
            lg, ids = eng.decode_checked([0, 1, 2, 3], torch.tensor(toks, dtype=torch.int32, device=dev),
                                         [37 + st] * 4, want_logits=True)
            res.append(lg.cpu().numpy())
            toks = [int(x) for x in ids.cpu().numpy()]
            if page and st == 0:
                # three writers copied the shared page; the last one kept it
                assert eng.pages_free() == free0 - 3
                t = [eng.page_table(r) for r in range(4)]
                assert len({int(x[2]) for x in t}) == 4 and all(np.array_equal(x[:2], t[0][:2]) for x in t)
        assert eng.sync() == 0, eng.last_error()
        outs[page] = (res, fed)
        eng.reset(-1)
        if page:
            assert eng.pages_free() == 4 * (128 // 16)
        eng.close()
    assert outs[0][1] == outs[16][1]
    for st, (a, b) in enumerate(zip(outs[0][0], outs[16][0])):
        assert np.array_equal(a, b), f"step {st}: forked rows differ between the cache layouts"
    # and a clone is right: row 2's own sequence through the oracle, step by step
    import oracle
    o = oracle.Model(s.replace(max_batch=1), W)
    o.prefill(0, prompt)
    res, fed = outs[16]
    for st in range(len(res)):
        lo, _ = o.decode_step([0], [fed[st][2]], [37 + st])
        check_logits(res[st][2], np.asarray(lo)[0], tolerance(s), f"clone row 2 step {st}")


def test_paged_fork_at_a_page_boundary(slm):
    """A source that ends exactly at a page boundary (32 positions, pages of 16): the
    clones share both full pages and there is no partial page to copy, so every row's first
    step takes a fresh page and nothing is copied; the rows then decode exactly as on a
    contiguous cache, and a clone matches the oracle."""
    s = synth.TINY.replace(max_batch=3, max_seq=96, kv_dtype=synth.DTYPE_BF16, dim=256, n_heads=4, n_kv_heads=1,
                           head_dim=64)
    W = synth.make_weights(s, seed=73)
    prompt = synth.make_prompt(s, 0, 32)
    dev = torch.device("cuda")
    outs = {}
    for page in (0, 16):
        eng = slm.Engine(s, W, kv_page_size=page)
        _, nid = eng.prefill_checked(0, prompt, want_logits=False)
        free0 = eng.pages_free()
        assert eng.fork(0, [1, 2]) == 0, eng.last_error()
        if page:
            assert eng.pages_free() == free0
            t0 = eng.page_table(0)
            assert all(np.array_equal(eng.page_table(r)[:2], t0[:2]) for r in (1, 2))
        toks = [(int(nid.item()) + 5 * r) % s.vocab for r in range(3)]
        res, fed = [], []
        for st in range(18):  # crosses into the fourth page at position 48
            fed.append(list(toks))
            lg, ids = eng.decode_checked([0, 1, 2], torch.tensor(toks, dtype=torch.int32, device=dev), [32 + st] * 3,
                                         want_logits=True)
            res.append(lg.cpu().numpy())
            toks = [int(x) for x in ids.cpu().numpy()]
            if page and st == 0:
                assert eng.pages_free() == free0 - 3  # one fresh page per row, no copies
                t = [eng.page_table(r) for r in range(3)]
                assert len({int(x[2]) for x in t}) == 3
        assert eng.sync() == 0, eng.last_error()
        outs[page] = (res, fed)
        eng.close()
    assert outs[0][1] == outs[16][1]
    for st, (a, b) in enumerate(zip(outs[0][0], outs[16][0])):
        assert np.array_equal(a, b), f"step {st}: forked rows differ between the cache layouts"
    import oracle
    o = oracle.Model(s.replace(max_batch=1), W)
    o.prefill(0, prompt)
    res, fed = outs[16]
    for st in range(len(res)):
        lo, _ = o.decode_step([0], [fed[st][1]], [32 + st])
        check_logits(res[st][1], np.asarray(lo)[0], tolerance(s), f"clone row 1 step {st}")


def test_paged_pool_exhaustion(slm):
    """A pool too small for every row: the step that needs a page no one has returns
    SLM_ECAPACITY and changes nothing; after a reset frees pages the same step runs,
    with the same results as on a contiguous cache."""
    s = synth.TINY.replace(max_batch=3, max_seq=96)
    W = synth.make_weights(s, seed=37)
    prompts = [synth.make_prompt(s, r, 30) for r in range(3)]
    eng = slm.Engine(s, W, kv_page_size=16, kv_pages=6)  # 2 pages per 30-token prompt
    dev = torch.device("cuda")
    for r in range(3):
        eng.prefill_checked(r, prompts[r], want_logits=False)
    assert eng.pages_free() == 0
    tok = torch.tensor([1, 2], dtype=torch.int32, device=dev)
    ids = torch.empty(2, dtype=torch.int32, device=dev)
    assert eng.decode_step([0, 1], tok, [30, 30], None, ids) == 0  # positions 30, 31 fit page 1
    assert eng.decode_step([0, 1], tok, [31, 31], None, ids) == 0
    rc = eng.decode_step([0, 1], tok, [32, 32], None, ids)  # both rows need a third page
    assert rc == slm.SLM_ECAPACITY, rc
    assert "page pool exhausted" in eng.last_error()
    assert eng.seq_len(0) == 32 and eng.seq_len(1) == 32
    eng.reset(2)
    assert eng.pages_free() == 2
    lg, _ = eng.decode_checked([0, 1], tok, [32, 32], want_logits=True)
    assert eng.sync() == 0, eng.last_error()
    ref = slm.Engine(s, W)
    for r in range(2):
        ref.prefill_checked(r, prompts[r], want_logits=False)
    for p in (30, 31):
        ref.decode_step([0, 1], tok, [p, p], None, ids)
    lg_ref, _ = ref.decode_checked([0, 1], tok, [32, 32], want_logits=True)
    assert np.array_equal(lg.cpu().numpy(), lg_ref.cpu().numpy())
    ref.close()
    eng.close()
