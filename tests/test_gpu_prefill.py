"""The tensor-core prefill (tcgen05 GEMMs + causal attention) against the oracle.

It is taken for prompts of 16 tokens or more when weights and KV cache are bf16; its
GEMM operands are bf16, so it is held to the bf16-cache tolerance (2e-2 * max|logit|).
Prompts longer than one 2048-position block exercise the chunked path, and decode
steps run on top of the cache it wrote.
"""
import numpy as np
import pytest

import oracle
import synth
from parity_util import check_id, check_logits

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

SHAPE = synth.Shape(dim=128, n_layers=2, n_heads=4, n_kv_heads=2, head_dim=64, hidden=256, vocab=512,
                    max_seq=2304, max_batch=2, rope_theta=10000.0, weight_dtype=synth.DTYPE_BF16,
                    kv_dtype=synth.DTYPE_BF16)


@pytest.fixture(scope="module")
def slm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import llama_decode_kv_gb300 as m
    return m


@pytest.mark.parametrize("n", [16, 100, 2100])
def test_tensor_prefill_matches_oracle(slm, n):
    s = SHAPE
    W = synth.make_weights(s, seed=21)
    prompt = synth.make_prompt(s, 3, n)
    o = oracle.Model(s, W)
    ref_logits, ref_id = o.prefill(0, prompt)
    eng = slm.Engine(s, W)
    lg, nid = eng.prefill_checked(0, prompt)
    check_logits(lg.cpu().numpy(), ref_logits, 2e-2, f"prefill n={n}")
    check_id(int(nid.item()), ref_logits, ref_id, f"prefill n={n}")
    # decode on top of the prefilled cache, teacher-forced with the oracle's ids
    tok = ref_id
    for st in range(4):
        rl, rid = o.decode_step([0], [tok], [n + st])
        gl, gid = eng.decode_checked([0], torch.tensor([tok], dtype=torch.int32, device="cuda"), [n + st])
        check_logits(gl[0].cpu().numpy(), rl[0], 2e-2, f"decode {st} after prefill n={n}")
        check_id(int(gid.item()), rl[0], int(rid[0]), f"decode {st} after prefill n={n}")
        tok = int(rid[0])
    assert eng.sync() == 0, eng.last_error()
    # the cache rows the prefill wrote, against the oracle's (bf16 values)
    for layer in (0, s.n_layers - 1):
        gk, gv = eng.kv(layer, 0)
        ok, ov = o.kv(layer, 0)
        assert gk.shape == ok.shape
        tol = 2e-2 * max(1.0, float(np.abs(ok).max()))
        assert np.abs(gk - ok).max() <= tol and np.abs(gv - ov).max() <= tol


@pytest.mark.parametrize("n_kv_heads", [1, 2])
def test_tensor_prefill_head_dim_128(slm, n_kv_heads):
    """head_dim 128: the attention kernel's 2-stage ring and the RoPE / append kernel's two
    pairs per lane and head; one prompt (two 64-row query blocks and a ragged third) and a
    batched call with three prompts, against the oracle."""
    s = SHAPE.replace(dim=256, n_heads=4, n_kv_heads=n_kv_heads, head_dim=128, max_seq=160, max_batch=3)
    W = synth.make_weights(s, seed=25)
    o = oracle.Model(s, W)
    prompt = synth.make_prompt(s, 1, 150)
    ref_logits, ref_id = o.prefill(0, prompt)
    eng = slm.Engine(s, W)
    lg, nid = eng.prefill_checked(0, prompt)
    check_logits(lg.cpu().numpy(), ref_logits, 2e-2, "hd128 prefill")
    check_id(int(nid.item()), ref_logits, ref_id, "hd128 prefill")
    gk, gv = eng.kv(s.n_layers - 1, 0)
    ok, ov = o.kv(s.n_layers - 1, 0)
    assert np.abs(gk - ok).max() <= 2e-2 * max(1.0, float(np.abs(ok).max()))
    assert np.abs(gv - ov).max() <= 2e-2 * max(1.0, float(np.abs(ov).max()))
    lens = [17, 64, 99]
    prompts = [synth.make_prompt(s, 4 + i, n) for i, n in enumerate(lens)]
    b = slm.Engine(s, W)
    dev = torch.device("cuda")
    toks = torch.as_tensor(np.concatenate(prompts).astype(np.int32)).to(dev)
    blg = torch.zeros((3, s.vocab), dtype=torch.float32, device=dev)
    ids = torch.zeros(3, dtype=torch.int32, device=dev)
    assert b.prefill_batch([0, 1, 2], toks, lens, blg, ids) == 0, b.last_error()
    assert b.sync() == 0, b.last_error()
    for i, p in enumerate(prompts):
        ref, rid = oracle.Model(s, W).prefill(0, p)
        check_logits(blg[i].cpu().numpy(), ref, 2e-2, f"hd128 batched prefill seq {i}")
        check_id(int(ids[i].item()), ref, rid, f"hd128 batched prefill seq {i}")
    eng.close()
    b.close()


def test_tensor_prefill_equals_token_by_token_prefill_closely(slm):
    # The same prompt through the tensor-core path (>= 16 tokens) and, token by token,
    # through the decode kernel (15 tokens then 1 decode step per further token).
    s = SHAPE
    W = synth.make_weights(s, seed=22)
    prompt = synth.make_prompt(s, 4, 40)
    a = slm.Engine(s, W)
    la, ia = a.prefill_checked(0, prompt)
    b = slm.Engine(s, W)
    b.prefill_checked(0, prompt[:15], want_logits=False)
    lb = None
    for p in range(15, 40):
        lb, ib = b.decode_checked([0], torch.tensor([int(prompt[p])], dtype=torch.int32, device="cuda"), [p])
    la, lb = la.cpu().numpy(), lb[0].cpu().numpy()
    assert np.abs(la - lb).max() <= 2e-2 * np.abs(lb).max()
    assert a.sync() == 0 and b.sync() == 0


def test_batched_prefill_equals_one_prefill_per_sequence(slm):
    # max_seq 128: prefill blocks of 128 rows, so the five prompts (318 positions) are cut
    # into three blocks with sequences crossing block edges
    s = SHAPE.replace(max_seq=128, max_batch=6)
    W = synth.make_weights(s, seed=31)
    seqs, lens = [4, 0, 2, 5, 1], [50, 90, 128, 17, 33]
    prompts = [synth.make_prompt(s, q, n) for q, n in zip(seqs, lens)]
    dev = torch.device("cuda")
    a = slm.Engine(s, W)
    toks = torch.as_tensor(np.concatenate(prompts).astype(np.int32)).to(dev)
    lg = torch.zeros((len(seqs), s.vocab), dtype=torch.float32, device=dev)
    ids = torch.zeros(len(seqs), dtype=torch.int32, device=dev)
    assert a.prefill_batch(seqs, toks, lens, lg, ids) == 0, a.last_error()
    assert a.sync() == 0, a.last_error()
    b = slm.Engine(s, W)
    for i, (q, p) in enumerate(zip(seqs, prompts)):
        lgb, nid = b.prefill_checked(q, p, want_logits=True)
        assert int(ids[i].item()) == int(nid.item())
        # the same GEMM rows, in other tiles: equal up to the order of fp32 sums
        np.testing.assert_allclose(lg[i].cpu().numpy(), lgb.cpu().numpy(), rtol=0, atol=1e-4)
        assert a.seq_len(q) == b.seq_len(q) == len(p)
        for layer in range(s.n_layers):
            ka, va = a.kv(layer, q)
            kb, vb = b.kv(layer, q)
            np.testing.assert_allclose(ka, kb, rtol=0, atol=1e-2 * np.abs(kb).max())
            np.testing.assert_allclose(va, vb, rtol=0, atol=1e-2 * np.abs(vb).max())
    assert b.sync() == 0
    # and against the oracle
    m = oracle.Model(s, W)
    for i, (q, p) in enumerate(zip(seqs, prompts)):
        ref, rid = m.prefill(q, p)
        check_logits(lg[i].cpu().numpy(), ref, 2e-2, f"batched prefill seq {q}")
        check_id(int(ids[i].item()), ref, rid, f"batched prefill seq {q}")
    a.close()
    b.close()


def test_batched_prefill_with_short_prompts(slm):
    """A batch holding prompts below the tensor-core minimum (1 and 15 tokens) beside
    longer ones (16, 70) takes the one-sequence-at-a-time path (token by token for the
    short prompts); every sequence's logits and id against the oracle, and a decode step
    on top of all four."""
    s = SHAPE.replace(max_seq=96, max_batch=4)
    W = synth.make_weights(s, seed=33)
    lens = [1, 15, 16, 70]
    prompts = [synth.make_prompt(s, 7 + i, n) for i, n in enumerate(lens)]
    dev = torch.device("cuda")
    eng = slm.Engine(s, W)
    toks = torch.as_tensor(np.concatenate(prompts).astype(np.int32)).to(dev)
    lg = torch.zeros((4, s.vocab), dtype=torch.float32, device=dev)
    ids = torch.zeros(4, dtype=torch.int32, device=dev)
    assert eng.prefill_batch([0, 1, 2, 3], toks, lens, lg, ids) == 0, eng.last_error()
    assert eng.sync() == 0, eng.last_error()
    m = oracle.Model(s, W)
    refs = []
    for i, p in enumerate(prompts):
        ref, rid = m.prefill(i, p)
        check_logits(lg[i].cpu().numpy(), ref, 2e-2, f"short-prompt batch seq {i}")
        check_id(int(ids[i].item()), ref, rid, f"short-prompt batch seq {i}")
        assert eng.seq_len(i) == lens[i]
        refs.append(rid)
    rl, rid = m.decode_step([0, 1, 2, 3], refs, lens)
    gl, gid = eng.decode_checked([0, 1, 2, 3], torch.tensor(refs, dtype=torch.int32, device=dev), lens)
    for i in range(4):
        check_logits(gl[i].cpu().numpy(), rl[i], 2e-2, f"decode after short-prompt batch, seq {i}")
        check_id(int(gid[i].item()), rl[i], int(rid[i]), f"decode after short-prompt batch, seq {i}")
    assert eng.sync() == 0
    eng.close()


def test_batched_prefill_refuses_bad_arguments(slm):
    s = SHAPE.replace(max_seq=64, max_batch=3)
    eng = slm.Engine(s, synth.make_weights(s, seed=3))
    dev = torch.device("cuda")
    toks = torch.zeros(64, dtype=torch.int32, device=dev)
    ids = torch.zeros(3, dtype=torch.int32, device=dev)
    EINVAL, ECAPACITY, ESTATE = -1, -3, -5
    assert eng.prefill_batch([0, 0], toks, [20, 20], None, ids) == EINVAL
    assert eng.prefill_batch([0, 3], toks, [20, 20], None, ids) == EINVAL
    assert eng.prefill_batch([0], toks, [65], None, ids) == ECAPACITY
    assert eng.prefill_batch([0], toks.cpu(), [20], None, ids) == EINVAL  # host tokens
    eng.prefill_checked(1, synth.make_prompt(s, 1, 20), want_logits=False)
    assert eng.prefill_batch([0, 1], toks, [20, 20], None, ids) == ESTATE
    assert eng.seq_len(0) == 0
    eng.close()


def test_batched_prefill_smol_16x512_equals_one_prefill_per_sequence(slm):
    """The batch-16 workload's prefill at full size: 16 SmolLM2-135M-shaped prompts of 512
    tokens (bf16 weights and cache) in one slm_prefill_batch call, i.e. one block of 8,192
    rows through every norm, GEMM, RoPE/append and attention launch, against one prefill
    per sequence (512-row blocks; the oracle pins that path on the small shapes above).
    Only the order of fp32 sums may differ (the norm kernels differ by block size), so the
    logits agree within the bf16-cache tolerance and the ids under the gap rule."""
    s = synth.SMOL.replace(max_seq=528, max_batch=16, kv_dtype=synth.DTYPE_BF16)
    W = synth.make_weights(s, seed=61)
    B, P = 16, 512
    prompts = [synth.make_prompt(s, r, P) for r in range(B)]
    dev = torch.device("cuda")
    a = slm.Engine(s, W)
    toks = torch.as_tensor(np.concatenate(prompts).astype(np.int32)).to(dev)
    lg = torch.zeros((B, s.vocab), dtype=torch.float32, device=dev)
    ids = torch.zeros(B, dtype=torch.int32, device=dev)
    assert a.prefill_batch(list(range(B)), toks, [P] * B, lg, ids) == 0, a.last_error()
    assert a.sync() == 0, a.last_error()
    lg, ids = lg.cpu().numpy(), ids.cpu().numpy()
    assert np.isfinite(lg).all()
    b = slm.Engine(s, W)
    for r in (0, 5, 15):
        lgb, nid = b.prefill_checked(r, prompts[r], want_logits=True)
        lgb = lgb.cpu().numpy()
        check_logits(lg[r], lgb, 2e-2, f"batched vs single prefill, seq {r}")
        check_id(int(ids[r]), lgb, int(nid.item()), f"batched vs single prefill, seq {r}")
        for layer in (0, s.n_layers - 1):
            ka, va = a.kv(layer, r)
            kb, vb = b.kv(layer, r)
            assert ka.shape == kb.shape == (s.n_kv_heads, P, s.head_dim)
            assert np.abs(ka - kb).max() <= 2e-2 * np.abs(kb).max()
            assert np.abs(va - vb).max() <= 2e-2 * np.abs(vb).max()
    assert b.sync() == 0
    a.close()
    b.close()
