"""slm_attention_decode (the split-K GQA decode attention on its own) against the
oracle's attention, from small ragged cases up to the long-context shape (4 rows x 32k
cached positions, Llama-3.2-1B heads)."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def slm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import llama_decode_kv_gb300 as m
    return m


def _inputs(B, H, KV, hd, cap, bf16, seed, qscale=2.0):
    rng = np.random.default_rng(seed)
    q = (rng.standard_normal((B, H, hd), dtype=np.float32) * np.float32(qscale))
    k = rng.standard_normal((B, KV, cap, hd), dtype=np.float32)
    v = rng.standard_normal((B, KV, cap, hd), dtype=np.float32)
    if bf16:
        kb, vb = synth.f32_to_bf16_rne(k), synth.f32_to_bf16_rne(v)
        k_ref, v_ref = synth.bf16_to_f32(kb), synth.bf16_to_f32(vb)
        k_dev = torch.from_numpy(kb.view(np.int16)).cuda()
        v_dev = torch.from_numpy(vb.view(np.int16)).cuda()
    else:
        k_ref, v_ref = k, v
        k_dev, v_dev = torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda()
    return q, k_ref, v_ref, torch.from_numpy(q).cuda(), k_dev, v_dev


def _run(slm, q_dev, k_dev, v_dev, lens, bf16):
    B, H, hd = q_dev.shape
    KV = k_dev.shape[1]
    ws = torch.empty(slm.slm_attention_workspace_bytes(B, H, KV, hd), dtype=torch.uint8, device="cuda")
    out = torch.full((B, H, hd), float("nan"), device="cuda")
    rc = slm.attention_decode(q_dev, k_dev, v_dev, lens, out, ws, slm.SLM_BF16 if bf16 else slm.SLM_F32)
    assert rc == 0, slm.slm_last_error(None)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _check(out, q, k, v, lens, pairs):
    H, KV = q.shape[1], k.shape[1]
    for b, h in pairs:
        g = h // (H // KV)
        want = oracle.attend(q[b, h], k[b, g, :lens[b]], v[b, g, :lens[b]])
        scale = max(1e-3, float(np.abs(want).max()))
        assert np.allclose(out[b, h], want, rtol=1e-4, atol=2e-5 * scale), (b, h, lens[b])


@pytest.mark.parametrize("B,H,KV,hd,bf16,lens", [
    (1, 4, 2, 16, False, [1]),
    (3, 4, 2, 16, False, [1, 31, 33]),
    (2, 9, 3, 64, False, [261, 100]),
    (3, 12, 3, 64, True, [5, 640, 1024]),
    (2, 8, 1, 128, True, [97, 300]),
    (2, 6, 2, 24, False, [40, 2]),
    (4, 16, 2, 64, True, [4000, 1, 2049, 3000]),
])
def test_attention_op_matches_oracle(slm, B, H, KV, hd, bf16, lens):
    cap = max(lens) + 7
    q, k, v, qd, kd, vd = _inputs(B, H, KV, hd, cap, bf16, seed=sum(lens) + hd)
    out = _run(slm, qd, kd, vd, lens, bf16)
    assert not np.isnan(out).any()
    _check(out, q, k, v, lens, [(b, h) for b in range(B) for h in range(H)])


def test_attention_op_long_context_shape(slm):
    # Llama-3.2-1B heads (32 query / 8 kv, head_dim 64), 4 rows, bf16 cache of 32832
    # positions, contexts around 32k: sampled (row, head) pairs against the oracle.
    B, H, KV, hd, cap = 4, 32, 8, 64, 32832
    lens = [32832, 32769, 32800, 30001]
    q, k, v, qd, kd, vd = _inputs(B, H, KV, hd, cap, True, seed=32768, qscale=3.0)
    out = _run(slm, qd, kd, vd, lens, True)
    assert not np.isnan(out).any()
    rng = np.random.default_rng(1)
    pairs = [(b, int(h)) for b in range(B) for h in rng.choice(H, 3, replace=False)]
    _check(out, q, k, v, lens, pairs)


def test_attention_op_rejects_bad_arguments(slm):
    B, H, KV, hd = 2, 4, 2, 16
    q, k, v, qd, kd, vd = _inputs(B, H, KV, hd, 8, False, seed=0)
    out = torch.empty((B, H, hd), device="cuda")
    need = slm.slm_attention_workspace_bytes(B, H, KV, hd)
    ws = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    assert slm.attention_decode(qd, kd, vd, [3, 9], out, ws, slm.SLM_F32) == slm.SLM_EINVAL  # ctx > cap
    assert slm.attention_decode(qd, kd, vd, [0, 2], out, ws, slm.SLM_F32) == slm.SLM_EINVAL
    assert slm.attention_decode(qd, kd, vd, [3, 2], out, ws[: need - 1], slm.SLM_F32) == slm.SLM_EINVAL
    assert slm.attention_decode(qd, kd, vd, [3, 2], out, ws[1:], slm.SLM_F32) == slm.SLM_EINVAL
    assert b"workspace" in slm.slm_last_error(None)
    assert slm.attention_decode(qd, kd, vd, [3, 2], out, ws, slm.SLM_F32) == 0
    torch.cuda.synchronize()


@pytest.mark.parametrize("noalloc", [False, True])
def test_misaligned_cache_is_refused_before_launch(slm, noalloc):
    """Cache rows are read 16 bytes at a time: a cache pointer off a 16-byte boundary (an
    offset view of a larger buffer) is refused with SLM_EINVAL and nothing is launched."""
    B, H, KV, hd, cap = 1, 4, 2, 16, 8
    q = torch.zeros((B, H, hd), device="cuda")
    base = torch.zeros(B * KV * cap * hd + 1, device="cuda")
    k = base[1:].view(B, KV, cap, hd)  # 4 bytes past an aligned address
    v = torch.zeros((B, KV, cap, hd), device="cuda")
    out = torch.full((B, H, hd), 7.0, device="cuda")
    if noalloc:
        rc = slm.attention_decode_noalloc(q, k, v, [cap], out, slm.SLM_F32)
    else:
        ws = torch.empty(slm.slm_attention_workspace_bytes(B, H, KV, hd), dtype=torch.uint8, device="cuda")
        rc = slm.attention_decode(q, k, v, [cap], out, ws, slm.SLM_F32)
    assert rc == slm.SLM_EINVAL
    assert b"16-byte aligned" in slm.slm_last_error(None)
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
