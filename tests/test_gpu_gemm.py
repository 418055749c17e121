"""The tensor-core GEMM tile (tcgen05 + TMA) against float64 matrix products of the
same bf16 values."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def slm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import llama_decode_kv_gb300 as m
    return m


@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (128, 128, 576), (300, 384, 576), (257, 200, 128),
                                   (1024, 3072, 2048), (64, 1536, 8192)])
def test_gemm_bf16_matches_fp64(slm, M, N, K):
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    a = synth.f32_to_bf16_rne(rng.standard_normal((M, K), dtype=np.float32))
    b = synth.f32_to_bf16_rne(rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02))
    ad = torch.from_numpy(a.view(np.int16)).cuda()
    bd = torch.from_numpy(b.view(np.int16)).cuda()
    c = torch.full((M, N), float("nan"), device="cuda")
    rc = slm.slm_debug_gemm_bf16(M, N, K, ad.data_ptr(), bd.data_ptr(), c.data_ptr(), None)
    assert rc == 0, slm.slm_last_error(None)
    want = synth.bf16_to_f32(a).astype(np.float64) @ synth.bf16_to_f32(b).astype(np.float64).T
    got = c.cpu().numpy()
    scale = np.abs(synth.bf16_to_f32(a)).astype(np.float64) @ np.abs(synth.bf16_to_f32(b)).astype(np.float64).T
    assert not np.isnan(got).any()
    assert np.all(np.abs(got - want) <= 1e-5 * scale + 1e-6), float(np.abs(got - want).max())


def test_gemm_rejects_bad_k(slm):
    x = torch.zeros((128, 100), dtype=torch.int16, device="cuda")
    c = torch.zeros((128, 128), device="cuda")
    assert slm.slm_debug_gemm_bf16(128, 128, 100, x.data_ptr(), x.data_ptr(), c.data_ptr(), None) == slm.SLM_EINVAL
