"""The allocation-free decode-attention entry point.

Some callers cannot allocate device memory -- an application whose allocator reserves
all of it up front, or a latency-critical loop that must not call cudaMalloc (it can
synchronise the device).  slm_attention_decode_noalloc serves them: it keeps its split-K
scratch in a fixed array inside the library.  This file checks it against the
workspace entry point (slm_attention_decode) through the C ABI, on two calls in a row
with different shapes, and directly against the oracle's attention on sampled heads
(so the check does not rest on the other entry point alone), and that a shape too
large for the fixed array is refused.
It is collected last so that a failure here never hides the other tests.
"""
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


def _inputs(B, H, KV, hd, cap, bf16, seed):
    rng = np.random.default_rng(seed)
    q = torch.from_numpy(rng.standard_normal((B, H, hd), dtype=np.float32) * np.float32(2.0)).cuda()
    k = rng.standard_normal((B, KV, cap, hd), dtype=np.float32)
    v = rng.standard_normal((B, KV, cap, hd), dtype=np.float32)
    if bf16:
        k = torch.from_numpy(synth.f32_to_bf16_rne(k).view(np.int16)).cuda()
        v = torch.from_numpy(synth.f32_to_bf16_rne(v).view(np.int16)).cuda()
    else:
        k, v = torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda()
    return q, k, v


CASES = [  # (B, H, KV, hd, bf16, lens): the second reuses the array the first left behind
    (3, 12, 3, 64, True, [700, 5, 1500]),
    (2, 8, 2, 64, False, [33, 2000]),
]


def test_noalloc_matches_workspace_entry_point_on_two_calls(slm):
    outs, refs = [], []
    inputs = [_inputs(B, H, KV, hd, max(l) + 3, bf16, seed=i) for i, (B, H, KV, hd, bf16, l) in enumerate(CASES)]
    # two calls in a row on the same stream, no synchronisation between them
    for (B, H, KV, hd, bf16, lens), (q, k, v) in zip(CASES, inputs):
        out = torch.full((B, H, hd), float("nan"), device="cuda")
        dt = slm.SLM_BF16 if bf16 else slm.SLM_F32
        assert slm.attention_decode_noalloc(q, k, v, lens, out, dt) == 0, slm.slm_last_error(None)
        outs.append(out)
    for (B, H, KV, hd, bf16, lens), (q, k, v) in zip(CASES, inputs):
        ws = torch.empty(slm.slm_attention_workspace_bytes(B, H, KV, hd), dtype=torch.uint8, device="cuda")
        ref = torch.full((B, H, hd), float("nan"), device="cuda")
        dt = slm.SLM_BF16 if bf16 else slm.SLM_F32
        assert slm.attention_decode(q, k, v, lens, ref, ws, dt) == 0, slm.slm_last_error(None)
        refs.append(ref)
    torch.cuda.synchronize()
    for got, ref in zip(outs, refs):
        got, ref = got.cpu().numpy(), ref.cpu().numpy()
        assert not np.isnan(got).any()
        scale = float(np.abs(ref).max())
        assert np.allclose(got, ref, rtol=1e-4, atol=2e-5 * scale)
    # the oracle, on a few (row, head) pairs of each call (q used as given: RoPE applied)
    rng = np.random.default_rng(3)
    for (B, H, KV, hd, bf16, lens), (q, k, v), got in zip(CASES, inputs, outs):
        qh, kh, vh, gh = q.cpu().numpy(), k.cpu().numpy(), v.cpu().numpy(), got.cpu().numpy()
        if bf16:
            kh = synth.bf16_to_f32(kh.view(np.uint16))
            vh = synth.bf16_to_f32(vh.view(np.uint16))
        for b in range(B):
            for h in rng.choice(H, 2, replace=False):
                g = h // (H // KV)
                want = oracle.attend(qh[b, h], kh[b, g, :lens[b]], vh[b, g, :lens[b]])
                sc = max(1e-3, float(np.abs(want).max()))
                assert np.allclose(gh[b, h], want, rtol=1e-4, atol=2e-5 * sc), (b, h)


def test_noalloc_refuses_shapes_beyond_its_array(slm):
    B, H, KV, hd = 16, 32, 8, 64
    need = slm.slm_attention_workspace_bytes(B, H, KV, hd)
    assert need > slm.slm_attention_noalloc_max_bytes() == 4 << 20
    q = torch.zeros((B, H, hd), device="cuda")
    k = torch.zeros((B, KV, 4, hd), device="cuda")
    out = torch.zeros((B, H, hd), device="cuda")
    rc = slm.attention_decode_noalloc(q, k, k, [4] * B, out, slm.SLM_F32)
    assert rc == slm.SLM_EINVAL
    assert b"fixed scratch array" in slm.slm_last_error(None)
