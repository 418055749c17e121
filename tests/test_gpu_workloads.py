"""The full-size workloads on the GPU against the oracle's stored values.

The oracle needs too long at these sizes to run inside a test (about half an hour per
Llama-3.2-1B-shaped row), so `tests/golden/make_goldens.py` (which calls only the
oracle) stored, per checked row and step, the greedy id, the top-2 gap, max|logit|, the
top-8 logits and the logits at 64 fixed vocabulary indices, plus the whole logits
vector at a few steps (`full_steps`: the prefill, the first, a middle and the last
decode step).  The GPU runs the whole
workload -- every row of the batch, full prompt, every decode step, in the launch
configuration the benchmark uses -- with the checked rows fed the oracle's ids (teacher
forcing) and the others their own, and is compared on those stored values:
logits within tol * max|logit| (tol 2e-2: bf16 KV cache) -- over the whole vocabulary
at the `full_steps`, on the stored values elsewhere -- and ids equal wherever the
oracle's top-2 gap exceeds 1e-2.
"""
import functools
import os

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
GAP = 1e-2


@pytest.fixture(scope="module")
def slm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import llama_decode_kv_gb300 as m
    return m


@functools.lru_cache(maxsize=2)
def weights_for(kind: str):
    shape = synth.SMOL if kind == "smol" else synth.LLAMA1B
    return synth.make_weights(shape)


def golden(prefix, row):
    path = os.path.join(GOLDEN, f"{prefix}_row{row}.npz")
    if not os.path.exists(path):
        pytest.fail(f"missing {path}: run tests/golden/make_goldens.py")
    return dict(np.load(path))


def check_step(gpu_logits_sampled, gpu_top_vals, gpu_id, g, s, tol, what, gpu_full=None):
    """gpu_logits_sampled: GPU logits at g['sample_idx']; gpu_top_vals: GPU logits at the
    oracle's top-8 indices; gpu_full: the whole GPU vector, compared element by element
    when step s is one of the golden's full_steps."""
    scale = float(g["maxabs"][s])
    err = max(float(np.abs(gpu_logits_sampled - g["sampled"][s]).max()),
              float(np.abs(gpu_top_vals - g["top_val"][s]).max()))
    full = list(g["full_steps"]) if "full_steps" in g else []
    if s in full:
        assert gpu_full is not None, f"{what}: the whole vector is needed at step {s}"
        ref = g["full"][full.index(s)]
        assert gpu_full.shape == ref.shape
        assert float(np.abs(ref).max()) == scale
        err = max(err, float(np.abs(gpu_full.astype(np.float64) - ref.astype(np.float64)).max()))
    assert err <= tol * scale, f"{what}: max|d logit| {err:.3e} > {tol} * {scale:.3e}"
    want = int(g["ids"][s])
    if g["gap"][s] > GAP:
        assert gpu_id == want, f"{what}: id {gpu_id} != oracle {want} (gap {g['gap'][s]:.3g})"
    else:
        top = list(g["top_idx"][s])
        ok = (gpu_id in top and g["top_val"][s][top.index(gpu_id)] >= g["top_val"][s][0] - GAP) or \
             (gpu_id not in top and g["top_val"][s][-1] >= g["top_val"][s][0] - GAP)
        assert ok, f"{what}: id {gpu_id} is not within the gap of the oracle's best"
    return err / scale


def run_workload(slm, wl, kind, prefix, checked_rows, shape=None):
    s = shape or wl.shape
    W = weights_for(kind)
    gold = {r: golden(prefix, r) for r in checked_rows}
    for r, g in gold.items():
        assert str(g["weights_sha256"]) == synth.digest(W), "synthetic weights differ from the golden run's"
    prompts = [synth.make_prompt(s, r, wl.prompt_len) for r in range(wl.batch)]
    for r, g in gold.items():
        assert np.array_equal(g["prompt"][: wl.prompt_len], prompts[r])
    eng = slm.Engine(s, W)
    dev = torch.device("cuda")
    worst = 0.0
    cur = {}
    sidx = {r: torch.as_tensor(gold[r]["sample_idx"], device=dev, dtype=torch.long) for r in gold}
    tidx = {r: torch.as_tensor(gold[r]["top_idx"], device=dev, dtype=torch.long) for r in gold}
    for r in range(wl.batch):
        lg, nid = eng.prefill_checked(r, prompts[r], want_logits=r in gold)
        g_id = int(nid.item())
        if r in gold:
            worst = max(worst, check_step(lg[sidx[r]].cpu().numpy(), lg[tidx[r][0]].cpu().numpy(), g_id,
                                          gold[r], 0, 2e-2, f"{prefix} row {r} prefill", lg.cpu().numpy()))
            cur[r] = int(gold[r]["ids"][0])
        else:
            cur[r] = g_id
    seqs = list(range(wl.batch))
    for step in range(wl.decode_steps):
        toks = torch.tensor([cur[r] for r in seqs], dtype=torch.int32, device=dev)
        lg, ids = eng.decode_checked(seqs, toks, [wl.prompt_len + step] * wl.batch, want_logits=True)
        ids_h = ids.cpu().numpy()
        for i, r in enumerate(seqs):
            if r in gold:
                full = step + 1 in list(gold[r]["full_steps"])
                worst = max(worst, check_step(lg[i][sidx[r]].cpu().numpy(), lg[i][tidx[r][step + 1]].cpu().numpy(),
                                              int(ids_h[i]), gold[r], step + 1, 2e-2,
                                              f"{prefix} row {r} step {step}", lg[i].cpu().numpy() if full else None))
                cur[r] = int(gold[r]["ids"][step + 1])
            else:
                cur[r] = int(ids_h[i])
    assert eng.sync() == 0, eng.last_error()
    eng.close()
    return worst


@pytest.mark.slow
def test_smol_b16_workload(slm):
    """SmolLM2-135M shape, bf16 KV, 16 rows x (512-token prompt + 512 greedy steps)."""
    wl = synth.WORKLOADS["smol_b16"]
    worst = run_workload(slm, wl, "smol", "smol_b16", [0, 7, 15])
    assert worst < 2e-2


@pytest.mark.slow
def test_llama1b_b1_workload(slm):
    """Llama-3.2-1B shape, bf16 KV, 2048-token prompt + 256 greedy steps, batch 1."""
    wl = synth.WORKLOADS["llama1b_b1"]
    worst = run_workload(slm, wl, "llama", "llama1b", [0])
    assert worst < 2e-2


@pytest.mark.slow
def test_llama1b_b8_workload(slm):
    """Llama-3.2-1B shape, bf16 KV, 8 rows x (2048-token prompt + 256 greedy steps)."""
    wl = synth.WORKLOADS["llama1b_b8"]
    worst = run_workload(slm, wl, "llama", "llama1b", [0, 1])
    assert worst < 2e-2


@pytest.mark.slow
def test_llama1b_long_context_workload(slm):
    """Llama-3.2-1B shape, bf16 KV: 4 rows x (32768-token prompt + 64 greedy decode steps).

    The oracle cannot prefill 32k positions, so this checks what holds at any size:
    * the layer-0 keys and values at sampled prompt positions and at the first decoded
      position equal the oracle's (they depend only on the token and the position);
    * the first decode step at position 32768 (decode kernel, split-K attention over
      32k cached positions) agrees with a prefill of the 32769-token sequence (GEMM
      path) within the tolerance;
    * all 64 steps run with a clean status and finite logits.
    """
    wl = synth.WORKLOADS["llama1b_long"]
    s = wl.shape
    W = weights_for("llama")
    eng = slm.Engine(s, W)
    dev = torch.device("cuda")
    prompts = [synth.make_prompt(s, r, wl.prompt_len) for r in range(wl.batch)]
    first = []
    for r in range(wl.batch):
        lg, nid = eng.prefill_checked(r, prompts[r], want_logits=False)
        first.append(int(nid.item()))
    ref = oracle.Model(s.replace(max_batch=1, max_seq=8), W)
    rng = np.random.default_rng(5)
    for r in (0, 3):
        k, v = eng.kv(0, r)
        for p in sorted(rng.choice(wl.prompt_len, 6, replace=False).tolist()) + [0, wl.prompt_len - 1]:
            ko, vo = ref.layer0_kv(int(prompts[r][p]), p)
            assert np.abs(k[:, p] - ko).max() <= 2e-2 * max(1.0, np.abs(ko).max()), (r, p)
            assert np.abs(v[:, p] - vo).max() <= 2e-2 * max(1.0, np.abs(vo).max()), (r, p)
    cur = list(first)
    step_logits = None
    for step in range(wl.decode_steps):
        toks = torch.tensor(cur, dtype=torch.int32, device=dev)
        lg, ids = eng.decode_checked(list(range(wl.batch)), toks, [wl.prompt_len + step] * wl.batch, want_logits=True)
        if step == 0:
            step_logits = lg[0].cpu().numpy()
        assert torch.isfinite(lg).all()
        cur = [int(x) for x in ids.cpu().numpy()]
    assert eng.sync() == 0, eng.last_error()
    k, v = eng.kv(0, 1)
    # decoded positions: tokens are known only through the engine's ids; check the first
    ko, vo = ref.layer0_kv(first[1], wl.prompt_len)
    assert np.abs(k[:, wl.prompt_len] - ko).max() <= 2e-2 * max(1.0, np.abs(ko).max())
    eng.close()
    # the 32769-token prefill of row 0 (prompt + its first generated token)
    s2 = s.replace(max_batch=1)
    e2 = slm.Engine(s2, W)
    lg2, _ = e2.prefill_checked(0, np.concatenate([prompts[0], [first[0]]]).astype(np.int32))
    lg2 = lg2.cpu().numpy()
    assert np.abs(step_logits - lg2).max() <= 2e-2 * np.abs(lg2).max()
    assert e2.sync() == 0
    e2.close()


@pytest.mark.slow
@pytest.mark.parametrize("page", [0, 256])
def test_long_context_2layer_against_oracle(slm, page):
    """4 rows x (32768-token prompt + 8 greedy decode steps) with the Llama-3.2-1B attention
    geometry (32 query heads, 8 kv heads, head_dim 64, bf16 KV, theta 500000) in a 2-layer
    model small enough for the oracle to prefill offline (tests/golden/long2l_row*.npz).
    The prompts go through the batched tensor-core prefill, the steps through the decode
    kernel's split-K attention over 32k cached positions (long chunks per work item);
    every logit of every row and step is compared with the oracle's (teacher forcing),
    ids under the gap rule.  The invariant behind it: cached generation equals the plain
    recomputation (GOTOken, "About one token per second").  page = 256: the same on a
    paged cache of 256-position pages."""
    wl = synth.WORKLOADS["llama1b_long_2l"]
    s = wl.shape
    W = synth.make_weights(s)
    gold = {r: golden("long2l", r) for r in range(wl.batch)}
    for r, g in gold.items():
        assert str(g["weights_sha256"]) == synth.digest(W)
        assert list(g["full_steps"]) == list(range(wl.decode_steps + 1))
    prompts = [synth.make_prompt(s, r, wl.prompt_len) for r in range(wl.batch)]
    for r, g in gold.items():
        assert np.array_equal(g["prompt"], prompts[r])
    eng = slm.Engine(s, W, kv_page_size=page)
    dev = torch.device("cuda")
    toks = torch.as_tensor(np.concatenate(prompts).astype(np.int32), device=dev)
    last = torch.empty((wl.batch, s.vocab), dtype=torch.float32, device=dev)
    ids = torch.empty(wl.batch, dtype=torch.int32, device=dev)
    eng._check(eng.prefill_batch(list(range(wl.batch)), toks, [wl.prompt_len] * wl.batch, last, ids),
               "slm_prefill_batch")
    lg0 = last.cpu().numpy()
    ids0 = ids.cpu().numpy()
    worst = 0.0
    for r in range(wl.batch):
        g = gold[r]
        worst = max(worst, check_step(lg0[r][g["sample_idx"]], lg0[r][g["top_idx"][0]], int(ids0[r]), g, 0,
                                      2e-2, f"long2l row {r} prefill", lg0[r]))
    cur = [int(gold[r]["ids"][0]) for r in range(wl.batch)]
    for step in range(wl.decode_steps):
        t = torch.tensor(cur, dtype=torch.int32, device=dev)
        lg, nid = eng.decode_checked(list(range(wl.batch)), t, [wl.prompt_len + step] * wl.batch, want_logits=True)
        lgh = lg.cpu().numpy()
        nidh = nid.cpu().numpy()
        for r in range(wl.batch):
            g = gold[r]
            worst = max(worst, check_step(lgh[r][g["sample_idx"]], lgh[r][g["top_idx"][step + 1]], int(nidh[r]), g,
                                          step + 1, 2e-2, f"long2l row {r} step {step}", lgh[r]))
        cur = [int(gold[r]["ids"][step + 1]) for r in range(wl.batch)]
    assert eng.sync() == 0, eng.last_error()
    # single rows of the same sequences (the cluster kernel, when it serves this shape)
    for r in (0, 3):
        eng.reset(r)
        lgp, nid = eng.prefill_checked(r, prompts[r], want_logits=True)
        check_step(lgp.cpu().numpy()[gold[r]["sample_idx"]], lgp.cpu().numpy()[gold[r]["top_idx"][0]],
                   int(nid.item()), gold[r], 0, 2e-2, f"long2l row {r} single prefill", lgp.cpu().numpy())
        t = torch.tensor([int(gold[r]["ids"][0])], dtype=torch.int32, device=dev)
        lg1, nid1 = eng.decode_checked([r], t, [wl.prompt_len], want_logits=True)
        check_step(lg1[0].cpu().numpy()[gold[r]["sample_idx"]], lg1[0].cpu().numpy()[gold[r]["top_idx"][1]],
                   int(nid1[0].item()), gold[r], 1, 2e-2, f"long2l row {r} single step", lg1[0].cpu().numpy())
    assert eng.sync() == 0, eng.last_error()
    eng.close()
    assert worst < 2e-2
