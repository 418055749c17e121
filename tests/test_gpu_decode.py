"""GPU parity of the decode path against the CPU oracle (through the C ABI)."""
import numpy as np
import pytest

import oracle
import synth
from parity_util import (check_id, check_logits, compare_runs, gpu_teacher_forced, oracle_reference,
                         tolerance)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def slm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import llama_decode_kv_gb300 as m
    return m


def _engine(slm, shape, W):
    return slm.Engine(shape, W)


def test_tiny_workload_matches_oracle(slm):
    # 5-token prompt, 8 greedy tokens (GOTOken, "About one token per second")
    wl = synth.WORKLOADS["tiny"]
    s = wl.shape
    W = synth.make_weights(s)
    prompts = [synth.make_prompt(s, 0, wl.prompt_len)]
    ref_ids, ref_logits = oracle_reference(s, prompts, wl.decode_steps, [0])
    eng = _engine(slm, s, W)
    g_logits, g_ids = gpu_teacher_forced(eng, s, prompts, ref_ids, wl.decode_steps, 1, [0])
    worst = compare_runs(s, ref_ids, ref_logits, g_logits, g_ids, [0], "tiny")
    assert len(g_ids[0]) == 8
    assert worst < tolerance(s)
    # the KV cache holds what the oracle's cache holds, slot by slot
    o = oracle.Model(s, W)
    o.prefill(0, prompts[0])
    for st in range(wl.decode_steps):
        o.decode_step([0], [ref_ids[0][st]], [wl.prompt_len + st])
    for layer in range(s.n_layers):
        gk, gv = eng.kv(layer, 0)
        ok, ov = o.kv(layer, 0)
        assert gk.shape == ok.shape == (s.n_kv_heads, 12, s.head_dim)
        assert np.allclose(gk, ok, atol=1e-4 * max(1.0, np.abs(ok).max()))
        assert np.allclose(gv, ov, atol=1e-4 * max(1.0, np.abs(ov).max()))


VARIANTS = {
    "mqa": dict(n_kv_heads=1),
    "mha": dict(n_kv_heads=4),
    "gqa8": dict(n_heads=8, n_kv_heads=1, dim=128),
    "bf16_weights": dict(weight_dtype=synth.DTYPE_BF16),
    "bf16_kv": dict(kv_dtype=synth.DTYPE_BF16),
    "ragged_dims": dict(dim=72, n_heads=3, n_kv_heads=1, head_dim=24, hidden=100, vocab=333),
    "wide_head": dict(dim=256, n_heads=2, n_kv_heads=1, head_dim=128, hidden=300),
}


SINGLE_ROW_VARIANTS = dict(VARIANTS, fp32_weights_bf16_kv=dict(kv_dtype=synth.DTYPE_BF16))


@pytest.mark.parametrize("name", sorted(SINGLE_ROW_VARIANTS))
def test_shape_variants_single_row(slm, name):
    """Single-row steps (the cluster kernel: attention clusters per kv head, FFN clusters)
    on every head geometry, against the oracle, rows decoded one at a time with ragged
    contexts."""
    s = synth.TINY.replace(max_batch=3, max_seq=96, **SINGLE_ROW_VARIANTS[name])
    W = synth.make_weights(s, seed=13)
    lens = [2, 17, 45]
    prompts = [synth.make_prompt(s, r, lens[r]) for r in range(3)]
    steps = 5
    ref_ids, ref_logits = oracle_reference(s, prompts, steps, [0, 1, 2], seed=13)
    eng = _engine(slm, s, W)
    assert eng.cluster_plan() is not None, "single-row steps of this shape should run on the cluster kernel"
    tol = tolerance(s)
    dev = torch.device("cuda")
    for r in range(3):
        lg, nid = eng.prefill_checked(r, prompts[r], want_logits=True)
        check_logits(lg.cpu().numpy(), ref_logits[r][0], tol, f"{name} row {r} prefill")
        check_id(int(nid.item()), ref_logits[r][0], ref_ids[r][0], f"{name} row {r} prefill")
        for st in range(steps):
            tok = torch.tensor([ref_ids[r][st]], dtype=torch.int32, device=dev)
            lg, ids = eng.decode_checked([r], tok, [lens[r] + st], want_logits=True)
            check_logits(lg[0].cpu().numpy(), ref_logits[r][st + 1], tol, f"{name} row {r} step {st}")
            check_id(int(ids[0].item()), ref_logits[r][st + 1], ref_ids[r][st + 1], f"{name} row {r} step {st}")
    assert eng.sync() == 0, eng.last_error()
    # the appended slots hold the oracle's keys and values
    o = oracle.Model(s.replace(max_batch=1), W)
    o.prefill(0, prompts[2])
    for st in range(steps):
        o.decode_step([0], [ref_ids[2][st]], [lens[2] + st])
    for layer in range(s.n_layers):
        gk, gv = eng.kv(layer, 2)
        ok, ov = o.kv(layer, 0)
        atol = (2e-2 if s.kv_dtype == synth.DTYPE_BF16 else 1e-4)
        assert np.allclose(gk, ok, atol=atol * max(1.0, np.abs(ok).max()))
        assert np.allclose(gv, ov, atol=atol * max(1.0, np.abs(ov).max()))
    eng.close()


@pytest.mark.parametrize("name", sorted(VARIANTS))
def test_shape_variants_batched_ragged(slm, name):
    s = synth.TINY.replace(max_batch=3, max_seq=96, **VARIANTS[name])
    W = synth.make_weights(s, seed=11)
    lens = [3, 9, 40]  # ragged contexts, one spanning several attention chunks
    prompts = [synth.make_prompt(s, r, lens[r]) for r in range(3)]
    steps = 6
    ref_ids, ref_logits = oracle_reference(s, prompts, steps, [0, 1, 2], seed=11)
    eng = _engine(slm, s, W)
    g_logits, g_ids = gpu_teacher_forced(eng, s, prompts, ref_ids, steps, 3, [0, 1, 2])
    compare_runs(s, ref_ids, ref_logits, g_logits, g_ids, [0, 1, 2], name)


STREAM_VARIANTS = {k: VARIANTS[k] for k in ("mqa", "bf16_kv", "gqa8", "ragged_dims", "wide_head")}
STREAM_VARIANTS.update({
    # bf16 caches with head_dim >= 32 take the head-split reduction
    "bf16kv_hd64_g4": dict(kv_dtype=synth.DTYPE_BF16, dim=256, n_heads=4, n_kv_heads=1, head_dim=64),
    "bf16kv_hd128_g2": dict(kv_dtype=synth.DTYPE_BF16, dim=256, n_heads=4, n_kv_heads=2, head_dim=128),
    "bf16kv_hd32_g8": dict(kv_dtype=synth.DTYPE_BF16, dim=256, n_heads=8, n_kv_heads=1, head_dim=32),
    "bf16kv_hd48_g3": dict(kv_dtype=synth.DTYPE_BF16, dim=144, n_heads=3, n_kv_heads=1, head_dim=48),
})


@pytest.mark.parametrize("name", sorted(STREAM_VARIANTS))
def test_streamed_attention_chunks(slm, name, monkeypatch):
    """Attention chunks too long for one shared-memory copy stream through per-warp rings
    (the long-context path).  Forcing 96-position chunks (SLM_ATTN_CHUNK) that are never
    copied whole (SLM_ATTN_STAGE=0) at contexts of 70..210 gives several chunks per row,
    chunks that end mid-pass and chunks that end at the new position, on every head
    geometry; against the oracle."""
    monkeypatch.setenv("SLM_ATTN_CHUNK", "96")
    monkeypatch.setenv("SLM_ATTN_STAGE", "0")
    s = synth.TINY.replace(max_batch=3, max_seq=256, **STREAM_VARIANTS[name])
    W = synth.make_weights(s, seed=17)
    lens = [70, 131, 203]
    prompts = [synth.make_prompt(s, r, lens[r]) for r in range(3)]
    steps = 4
    ref_ids, ref_logits = oracle_reference(s, prompts, steps, [0, 1, 2], seed=17)
    eng = _engine(slm, s, W)
    g_logits, g_ids = gpu_teacher_forced(eng, s, prompts, ref_ids, steps, 3, [0, 1, 2])
    compare_runs(s, ref_ids, ref_logits, g_logits, g_ids, [0, 1, 2], name + " streamed")


def test_kv_slots_written_exactly(slm):
    s = synth.TINY.replace(max_batch=2)
    W = synth.make_weights(s, seed=5)
    eng = _engine(slm, s, W)
    sentinel = 12345.0
    eng.fill_kv(sentinel)
    p0 = synth.make_prompt(s, 0, 7)
    eng.prefill_checked(1, p0)
    before = [eng.kv(l, 1, n_pos=s.max_seq) for l in range(s.n_layers)]
    other = [eng.kv(l, 0, n_pos=s.max_seq) for l in range(s.n_layers)]
    for l in range(s.n_layers):
        k, v = before[l]
        assert np.all(k[:, 7:] == sentinel) and np.all(v[:, 7:] == sentinel)
        assert not np.any(k[:, :7] == sentinel)
        assert np.all(other[l][0] == sentinel)  # sequence 0 untouched
    tok = torch.tensor([int(p0[-1])], dtype=torch.int32, device="cuda")
    eng.decode_checked([1], tok, [7])
    for l in range(s.n_layers):
        k, v = eng.kv(l, 1, n_pos=s.max_seq)
        kb, vb = before[l]
        assert np.array_equal(k[:, :7], kb[:, :7]) and np.array_equal(v[:, :7], vb[:, :7])
        assert not np.any(k[:, 7] == sentinel)
        assert np.all(k[:, 8:] == sentinel) and np.all(v[:, 8:] == sentinel)
    # the new slot equals the oracle's layer-0 key/value for (token, position)
    o = oracle.Model(s, W)
    ko, vo = o.layer0_kv(int(p0[-1]), 7)
    k, v = eng.kv(0, 1, n_pos=8)
    assert np.allclose(k[:, 7], ko, atol=1e-5) and np.allclose(v[:, 7], vo, atol=1e-5)


def test_api_errors_on_device(slm):
    s = synth.TINY.replace(max_batch=2, max_seq=16)
    eng = _engine(slm, s, synth.make_weights(s))
    p = synth.make_prompt(s, 0, 5)
    eng.prefill_checked(0, p)
    tok = torch.tensor([1, 2], dtype=torch.int32, device="cuda")
    ids = torch.empty(2, dtype=torch.int32, device="cuda")
    assert eng.prefill(0, torch.tensor(p, device="cuda"), None, ids[:1]) == slm.SLM_ESTATE
    assert eng.decode_step([0], tok[:1], [4], None, ids) == slm.SLM_EPOS
    assert eng.decode_step([0, 0], tok, [5, 5], None, ids) == slm.SLM_EINVAL
    assert eng.decode_step([0, 1], tok, [5, 0], None, ids) == slm.SLM_OK
    assert eng.seq_len(0) == 6 and eng.seq_len(1) == 1
    bad = np.array([s.vocab], dtype=np.int32)  # host token: checked on the host
    assert eng.decode_step([0], bad, [6], None, ids) == slm.SLM_EINVAL
    eng.reset(1)
    assert eng.seq_len(1) == 0
    eng.reset(0)
    eng.prefill_checked(0, synth.make_prompt(s, 1, s.max_seq))
    assert eng.decode_step([0], tok[:1], [s.max_seq], None, ids) == slm.SLM_ECAPACITY
    # a device token out of range is caught on the device and reported by slm_sync
    eng.reset(-1)
    eng.prefill_checked(0, p)
    badd = torch.tensor([s.vocab + 5], dtype=torch.int32, device="cuda")
    assert eng.decode_step([0], badd, [5], None, ids) == slm.SLM_OK
    assert eng.sync() == slm.SLM_EDEVICE
    # the context keeps working afterwards
    eng.reset(-1)
    eng.prefill_checked(0, p)
    assert eng.decode_step([0], tok[:1], [5], None, ids) == slm.SLM_OK
    assert eng.sync() == slm.SLM_OK


@pytest.mark.parametrize("batch", [1, 2])
def test_decode_into_the_last_cache_slot(slm, batch):
    """Prompts that leave a few free positions (tensor-core prefill, bf16 weights and
    cache), then decode steps up to the last slot, max_seq - 1, against the oracle (one
    row: the cluster kernel; two rows: the persistent kernel); one more step is refused
    with SLM_ECAPACITY and changes nothing."""
    s = synth.TINY.replace(max_batch=batch, max_seq=64, weight_dtype=synth.DTYPE_BF16, kv_dtype=synth.DTYPE_BF16,
                           dim=256, n_heads=4, n_kv_heads=1, head_dim=64)
    W = synth.make_weights(s, seed=71)
    lens = [60, 57][:batch]
    prompts = [synth.make_prompt(s, r, lens[r]) for r in range(batch)]
    steps = 4  # row 0 decodes positions 60..63
    rows = list(range(batch))
    ref_ids, ref_logits = oracle_reference(s, prompts, steps, rows, seed=71)
    eng = _engine(slm, s, W)
    if batch == 1:
        assert eng.cluster_plan() is not None
    g_logits, g_ids = gpu_teacher_forced(eng, s, prompts, ref_ids, steps, batch, rows)
    compare_runs(s, ref_ids, ref_logits, g_logits, g_ids, rows, f"last slot, batch {batch}")
    assert eng.seq_len(0) == s.max_seq
    tok = torch.tensor([1], dtype=torch.int32, device="cuda")
    ids = torch.empty(1, dtype=torch.int32, device="cuda")
    assert eng.decode_step([0], tok, [s.max_seq], None, ids) == slm.SLM_ECAPACITY
    assert eng.seq_len(0) == s.max_seq
    assert eng.sync() == 0, eng.last_error()
    eng.close()


def test_host_buffers_give_the_same_results(slm):
    s = synth.TINY.replace(max_batch=2)
    W = synth.make_weights(s, seed=3)
    a = _engine(slm, s, W)
    b = _engine(slm, s, W)
    p = [synth.make_prompt(s, r, 6) for r in range(2)]
    for r in range(2):
        la = np.empty(s.vocab, np.float32)
        ia = np.empty(1, np.int32)
        assert a.prefill(r, p[r], la, ia) == 0          # host buffers: synchronous
        lb, ib = b.prefill_checked(r, p[r])
        assert np.array_equal(la, lb.cpu().numpy()) and ia[0] == int(ib.item())
    toks = np.array([1, 2], np.int32)
    la = np.empty((2, s.vocab), np.float32)
    ia = np.empty(2, np.int32)
    assert a.decode_step([0, 1], toks, [6, 6], la, ia) == 0
    lb, ib = b.decode_checked([0, 1], torch.tensor(toks, device="cuda"), [6, 6])
    assert np.array_equal(la, lb.cpu().numpy()) and np.array_equal(ia, ib.cpu().numpy())


def test_decode_from_empty_sequence_equals_prefill(slm):
    # decoding position 0 of an empty sequence is a one-token prompt
    s = synth.TINY
    W = synth.make_weights(s)
    a = _engine(slm, s, W)
    b = _engine(slm, s, W)
    la, ia = a.prefill_checked(0, np.array([17], np.int32))
    lb, ib = b.decode_checked([0], torch.tensor([17], dtype=torch.int32, device="cuda"), [0])
    assert np.array_equal(la.cpu().numpy(), lb[0].cpu().numpy())


@pytest.mark.slow
def test_smol_b1_workload_full(slm):
    """SmolLM2-135M shape, batch 1, 5-token prompt, 256 greedy decode steps, fp32 KV."""
    wl = synth.WORKLOADS["smol_b1"]
    s = wl.shape
    W = synth.make_weights(s)
    prompts = [synth.make_prompt(s, 0, wl.prompt_len)]
    ref_ids, ref_logits = oracle_reference(s, prompts, wl.decode_steps, [0])
    eng = _engine(slm, s, W)
    g_logits, g_ids = gpu_teacher_forced(eng, s, prompts, ref_ids, wl.decode_steps, 1, [0])
    compare_runs(s, ref_ids, ref_logits, g_logits, g_ids, [0], "smol_b1")


@pytest.mark.parametrize("name,batch", [("bf16_tc_b13", 13), ("bf16_tc_b16_bf16kv", 16)])
def test_batch16_tensor_core_path(slm, name, batch):
    # batches of 9..16 rows with bf16 weights run the GEMV phases and the logits on the
    # tensor cores (activations as bf16 hi + lo planes); ragged contexts
    kv = synth.DTYPE_BF16 if "bf16kv" in name else synth.DTYPE_F32
    s = synth.TINY.replace(max_batch=16, max_seq=96, weight_dtype=synth.DTYPE_BF16, kv_dtype=kv,
                           dim=128, n_heads=4, n_kv_heads=2, head_dim=32, hidden=200, vocab=300)
    W = synth.make_weights(s, seed=13)
    lens = [3 + (7 * r) % 40 for r in range(batch)]
    prompts = [synth.make_prompt(s, r, lens[r]) for r in range(batch)]
    steps = 4
    rows = list(range(batch))
    ref_ids, ref_logits = oracle_reference(s, prompts, steps, rows, seed=13)
    eng = _engine(slm, s, W)
    g_logits, g_ids = gpu_teacher_forced(eng, s, prompts, ref_ids, steps, batch, rows)
    compare_runs(s, ref_ids, ref_logits, g_logits, g_ids, rows, name)


def test_batch16_tensor_core_k_split(slm):
    # hidden 2048: at 16 padded rows W2's input does not fit the activation tile in one
    # piece, so the tensor-core residual epilogue accumulates over K tiles
    s = synth.TINY.replace(max_batch=16, max_seq=64, weight_dtype=synth.DTYPE_BF16, kv_dtype=synth.DTYPE_F32,
                           dim=128, n_heads=4, n_kv_heads=2, head_dim=32, hidden=2048, vocab=300)
    W = synth.make_weights(s, seed=17)
    batch = 12
    lens = [2 + (5 * r) % 23 for r in range(batch)]
    prompts = [synth.make_prompt(s, r, lens[r]) for r in range(batch)]
    steps = 3
    rows = list(range(batch))
    ref_ids, ref_logits = oracle_reference(s, prompts, steps, rows, seed=17)
    eng = _engine(slm, s, W)
    g_logits, g_ids = gpu_teacher_forced(eng, s, prompts, ref_ids, steps, batch, rows)
    compare_runs(s, ref_ids, ref_logits, g_logits, g_ids, rows, "bf16_tc_ksplit")


def test_one_engine_serves_every_batch_size(slm):
    # a max_batch 16 engine: steps of 1, 5 and 16 rows run the 1-, 8- and 16-row kernels
    # (CUDA-core and tensor-core GEMVs) over the same weight layout and caches
    s = synth.TINY.replace(max_batch=16, max_seq=64, weight_dtype=synth.DTYPE_BF16, kv_dtype=synth.DTYPE_BF16,
                           dim=128, n_heads=4, n_kv_heads=2, head_dim=32, hidden=256, vocab=300)
    W = synth.make_weights(s, seed=23)
    rows = list(range(16))
    lens = [4 + (3 * r) % 17 for r in rows]
    prompts = [synth.make_prompt(s, r, lens[r]) for r in rows]
    steps = 3
    ref_ids, ref_logits = oracle_reference(s, prompts, 3 * steps, rows, seed=23)
    eng = _engine(slm, s, W)
    dev = torch.device("cuda")
    g_logits = {r: [] for r in rows}
    g_ids = {r: [] for r in rows}
    cur = {}
    for r in rows:
        lg, nid = eng.prefill_checked(r, prompts[r], want_logits=True)
        g_logits[r].append(lg.cpu().numpy())
        g_ids[r].append(int(nid.item()))
        cur[r] = ref_ids[r][0]
    done = {r: 0 for r in rows}
    # every row takes 3 * steps decode steps, in batches of 1, 5 and 16 rows in turn
    k = 0
    while any(done[r] < 3 * steps for r in rows):
        width = (1, 5, 16)[k % 3]
        k += 1
        seqs = sorted((r for r in rows if done[r] < 3 * steps), key=lambda r: (done[r], r))[:width]
        toks = torch.tensor([cur[r] for r in seqs], dtype=torch.int32, device=dev)
        lg, nid = eng.decode_checked(seqs, toks, [lens[r] + done[r] for r in seqs], want_logits=True)
        lg, nid = lg.cpu().numpy(), nid.cpu().numpy()
        for i, r in enumerate(seqs):
            done[r] += 1
            g_logits[r].append(lg[i])
            g_ids[r].append(int(nid[i]))
            if done[r] < 3 * steps:
                cur[r] = ref_ids[r][done[r]]
    assert all(v == 3 * steps for v in done.values())
    assert eng.sync() == 0, eng.last_error()
    compare_runs(s, ref_ids, ref_logits, g_logits, g_ids, rows, "mixed batch sizes")
    eng.close()
