"""On-device sampling (slm_sample) against the sampling oracle on identical logits and
uniforms.  The drawn id is unique once the uniform is not at a boundary of the
cumulative distribution (and top-p not at a boundary of the cut): top-k draws keep the
uniform clear of the boundaries and must give the oracle's id; over the whole vocabulary
(boundaries ~1e-5 apart) the id must hold the uniform inside its interval up to the
rounding of the running sums, and equal the oracle's where the uniform is clear."""
import numpy as np
import pytest
import torch

from oracle import sampling

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def slm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import llama_decode_kv_gb300 as m
    return m


def _safe_uniform(rng, x, T, k, p):
    """A uniform clear of every CDF boundary by min(1e-3, 0.2 / candidates) of the total
    (far above the rounding of fp32 running sums over at most 1024 candidates)."""
    if T == 0.0:
        return float(rng.random())
    _, w = sampling.candidates(x, T, k, p)
    F = np.cumsum(np.array(w, dtype=np.float64))
    F /= F[-1]
    margin = min(1e-3, 0.2 / len(w))
    for _ in range(1000):
        u = float(rng.random())
        if np.min(np.abs(F - u)) > margin:
            return u
    raise AssertionError("no safe uniform")


def _cut_is_safe(x, T, k, p):
    if p >= 1.0 or T == 0.0:
        return True
    _, w = sampling.candidates(x, T, k, 1.0)
    F = np.cumsum(np.array(w, dtype=np.float64))
    F /= F[-1]
    return np.min(np.abs(F - p)) > 1e-4


def _run(slm, logits, T, k, p, us):
    dev = torch.device("cuda")
    lg = torch.as_tensor(logits, dtype=torch.float32).to(dev)
    u = torch.as_tensor(np.array(us, dtype=np.float32)).to(dev)
    ids = torch.full((logits.shape[0],), -7, dtype=torch.int32, device=dev)
    rc = slm.sample(lg, T, k, p, u, ids)
    assert rc == 0, slm.slm_last_error(None)
    torch.cuda.synchronize()
    return ids.cpu().numpy()


CASES = [
    (1000, 0.0, 0, 1.0),
    (1000, 0.8, 40, 1.0),
    (1000, 0.8, 40, 0.95),
    (5000, 1.3, 1024, 0.9),
    (5000, 1.0, 0, 1.0),
    (3000, 0.5, 1, 1.0),
    (49152, 0.8, 40, 0.95),
    (128256, 1.0, 0, 1.0),
    (128256, 0.7, 50, 0.9),
]


def _check(x, T, k, p, u, g, delta=1e-5):
    """g is a valid draw for u: u lies in g's interval of the oracle's CDF, up to delta
    (rounding of the running sums); it is the oracle's draw when u is further than
    2 * delta from every boundary."""
    want = sampling.sample(x, T, k, p, u)
    if T == 0.0:
        assert g == want
        return
    order, w = sampling.candidates(x, T, k, p)
    F = np.cumsum(np.array(w, dtype=np.float64))
    F /= F[-1]
    assert g in order, (g, "not a candidate")
    j = order.index(g)
    lo = F[j - 1] if j else 0.0
    assert lo - delta <= u <= F[j] + delta, (g, want, u, lo, F[j])
    if np.min(np.abs(F - u)) > 2 * delta:
        assert g == want


@pytest.mark.parametrize("V,T,k,p", CASES)
def test_sampling_matches_the_oracle(slm, V, T, k, p):
    rng = np.random.default_rng(V * 7 + k)
    B = 6
    logits = rng.normal(0, 2.0, (B, V)).astype(np.float32)
    us = []
    for b in range(B):
        while not _cut_is_safe(logits[b], T, k, p):
            logits[b] = rng.normal(0, 2.0, V).astype(np.float32)
        # top-k: a uniform well clear of the (few) boundaries; the whole vocabulary has
        # boundaries ~1e-5 apart, so any uniform
        us.append(_safe_uniform(rng, logits[b], T, k, p) if k >= 1 else float(rng.random()))
    got = _run(slm, logits, T, k, p, us)
    for b in range(B):
        _check(logits[b], T, k, p, us[b], int(got[b]))
    if k >= 1 or T == 0.0:
        assert list(got) == [sampling.sample(logits[b], T, k, p, us[b]) for b in range(B)]


def test_ties_at_the_top_k_threshold_take_the_lowest_indices(slm):
    # integer logits in a small range: thousands of equal values at the k-th largest
    rng = np.random.default_rng(3)
    B, V = 4, 4096
    logits = rng.integers(0, 6, (B, V)).astype(np.float32)
    for (T, k, p) in ((1.0, 100, 1.0), (0.6, 37, 0.8), (0.0, 0, 1.0), (2.0, 1024, 1.0)):
        us = [_safe_uniform(rng, logits[b], T, k, p) for b in range(B)]
        got = _run(slm, logits, T, k, p, us)
        want = [sampling.sample(logits[b], T, k, p, us[b]) for b in range(B)]
        assert list(got) == want, (T, k, p)


def test_edge_sizes(slm):
    rng = np.random.default_rng(11)
    one = np.array([[0.3]], dtype=np.float32)
    for (T, k, p) in ((0.0, 0, 1.0), (1.0, 0, 1.0), (1.0, 5, 0.5)):
        assert list(_run(slm, one, T, k, p, [0.99])) == [0]
    x = rng.normal(0, 1, (1, 7)).astype(np.float32)
    u = _safe_uniform(rng, x[0], 1.0, 100, 1.0)  # k above the vocabulary: all of it, sorted
    assert list(_run(slm, x, 1.0, 100, 1.0, [u])) == [sampling.sample(x[0], 1.0, 100, 1.0, u)]


def test_sampling_from_decode_step_logits(slm):
    import synth
    s = synth.SMOL.replace(max_batch=4, max_seq=64, n_layers=2)
    eng = slm.Engine(s, synth.make_weights(s, seed=2))
    for r in range(4):
        eng.prefill_checked(r, synth.make_prompt(s, r, 6), want_logits=False)
    toks = torch.tensor([5, 17, 300, 4000], dtype=torch.int32, device="cuda")
    lg, _ = eng.decode_checked([0, 1, 2, 3], toks, [6] * 4, want_logits=True)
    host = lg.cpu().numpy()
    rng = np.random.default_rng(9)
    us = [_safe_uniform(rng, host[b], 0.8, 40, 0.95) for b in range(4)]
    u = torch.as_tensor(np.array(us, dtype=np.float32)).cuda()
    ids = torch.empty(4, dtype=torch.int32, device="cuda")
    assert slm.sample(lg, 0.8, 40, 0.95, u, ids) == 0
    assert list(ids.cpu().numpy()) == [sampling.sample(host[b], 0.8, 40, 0.95, us[b]) for b in range(4)]
    eng.close()


def test_bad_arguments_are_refused(slm):
    dev = torch.device("cuda")
    lg = torch.zeros((2, 10), device=dev)
    u = torch.zeros(2, device=dev)
    ids = torch.zeros(2, dtype=torch.int32, device=dev)
    EINVAL = -1
    assert slm.sample(lg, 1.0, 2000, 1.0, u, ids) == EINVAL
    assert slm.sample(lg, 1.0, 5, 0.0, u, ids) == EINVAL
    assert slm.sample(lg, 1.0, 0, 0.9, u, ids) == EINVAL
    assert slm.sample(lg, -1.0, 5, 1.0, u, ids) == EINVAL
    assert slm.sample(lg, float("inf"), 5, 1.0, u, ids) == EINVAL
    assert slm.sample(lg.cpu(), 1.0, 5, 1.0, u, ids) == EINVAL  # host logits
