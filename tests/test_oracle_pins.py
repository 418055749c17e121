"""Pins for the CPU oracle: each test ties one of its pieces to something other than
itself -- a value or invariant the pages state, a closed form, or brute force in float64
on tiny inputs -- so that a dropped term, a wrong sign, a wrong index or a transposed
operand in ``oracle/oracle.c`` fails at least one of them.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import DTYPE_BF16, DTYPE_F32

RNG = np.random.default_rng(20261202)


# ----------------------------------------------------------------------------- bf16

def test_bf16_upcast_is_a_16_bit_shift():
    # GOTOken, "Loading the model and tokenizer": bf16 is the top 16 bits of an fp32
    # word, so widening is a left shift by 16.
    assert oracle.bf16_up(0x3F80) == 1.0
    assert oracle.bf16_up(0xC000) == -2.0
    assert oracle.bf16_up(0x4049) == np.float32(3.140625)
    assert oracle.bf16_up(0x0000) == 0.0
    for b in RNG.integers(0, 0x7F80, 50):
        want = np.array([int(b) << 16], dtype=np.uint32).view(np.float32)[0]
        assert oracle.bf16_up(int(b)) == want


def test_bf16_round_nearest_even():
    one = 1.0
    cases = [
        (one, one),
        (one + 2.0 ** -8, one),                          # halfway, even neighbour below
        (one + 3 * 2.0 ** -8, one + 2.0 ** -6),          # halfway, even neighbour above
        (one + 2.0 ** -8 + 2.0 ** -20, one + 2.0 ** -7),  # just above halfway
        (-(one + 2.0 ** -8), -one),
        (3.14159265, 3.140625),
    ]
    got = oracle.bf16_round(np.array([c[0] for c in cases], dtype=np.float32))
    assert list(got) == [np.float32(c[1]) for c in cases]
    # every result has its low 16 bits clear and lies within half an ulp (2^-8 rel.)
    x = (RNG.standard_normal(1000) * 10).astype(np.float32)
    r = oracle.bf16_round(x)
    assert np.all(r.view(np.uint32) & 0xFFFF == 0)
    assert np.all(np.abs(r - x) <= np.abs(x) * 2.0 ** -8 * 1.0000001)


# ----------------------------------------------------------------------------- matvec

def test_matvec_small_integers_exact():
    # integer products and sums below 2^24 are exact in fp32: the result must be the
    # exact integer matrix-vector product (catches a transposed or misindexed W).
    w = RNG.integers(-8, 9, (7, 13)).astype(np.float32)
    x = RNG.integers(-8, 9, 13).astype(np.float32)
    got = oracle.matvec(w, x)
    want = (w.astype(np.int64) @ x.astype(np.int64)).astype(np.float32)
    assert np.array_equal(got, want)


def test_matvec_within_fp32_bound_of_fp64():
    n_in, n_out = 576, 97
    w = RNG.standard_normal((n_out, n_in)).astype(np.float32)
    x = RNG.standard_normal(n_in).astype(np.float32)
    got = oracle.matvec(w, x).astype(np.float64)
    exact = w.astype(np.float64) @ x.astype(np.float64)
    bound = n_in * 2.0 ** -24 * (np.abs(w).astype(np.float64) @ np.abs(x).astype(np.float64))
    assert np.all(np.abs(got - exact) <= bound)


def test_matvec_matches_same_order_fp32_replay():
    # GOTOken, "Building it one piece at a time": an fp32 replay of the loop in the same
    # rounding order matched all 576 query-projection outputs bit for bit.  Replay
    # acc = fl(acc + fl(w*x)) with numpy float32 scalars (one rounding per operation).
    n_in, n_out = 576, 576
    w = RNG.standard_normal((n_out, n_in)).astype(np.float32) * np.float32(0.02)
    x = RNG.standard_normal(n_in).astype(np.float32)
    got = oracle.matvec(w, x)
    rows = RNG.choice(n_out, 24, replace=False)
    for i in rows:
        acc = np.float32(0.0)
        for j in range(n_in):
            acc = np.float32(acc + np.float32(w[i, j] * x[j]))
        assert got[i] == acc


# ----------------------------------------------------------------------------- rmsnorm

def test_rmsnorm_closed_forms():
    n = 576
    eps = 1e-5
    # constant vector: x * rsqrt(c^2 + eps) * g
    for c in (0.5, -3.0, 1e-3):
        x = np.full(n, c, dtype=np.float32)
        g = RNG.standard_normal(n).astype(np.float32)
        got = oracle.rmsnorm(x, g, eps)
        want = c / np.sqrt(c * c + eps) * g.astype(np.float64)
        assert np.allclose(got, want, rtol=1e-6, atol=1e-7)
    # unit gains and eps=0 -> mean square of the output is 1
    x = RNG.standard_normal(n).astype(np.float32) * 7
    got = oracle.rmsnorm(x, np.ones(n, np.float32), 0.0).astype(np.float64)
    assert abs(np.mean(got ** 2) - 1.0) < 1e-5
    # against the float64 formula with non-uniform gains
    g = RNG.standard_normal(n).astype(np.float32)
    got = oracle.rmsnorm(x, g, eps).astype(np.float64)
    x64 = x.astype(np.float64)
    want = x64 / np.sqrt(np.mean(x64 ** 2) + eps) * g
    assert np.allclose(got, want, rtol=1e-5, atol=1e-6)


# ----------------------------------------------------------------------------- RoPE

def test_rope_identity_at_position_zero():
    v = RNG.standard_normal(4 * 64).astype(np.float32)
    assert np.array_equal(oracle.rope(v, 4, 64, 0, 10000.0), v)


def test_rope_rotates_half_split_pairs_with_theta_frequencies():
    # unit vector e_i goes to cos(a) e_i + sin(a) e_{i+hd/2}, a = pos * theta^(-2i/hd)
    hd, theta = 64, 100000.0
    for i in (0, 1, 7, 31):
        for pos in (1, 5, 1000, 32767):
            v = np.zeros(hd, np.float32)
            v[i] = 1.0
            got = oracle.rope(v, 1, hd, pos, theta)
            a = pos * theta ** (-2.0 * i / hd)
            want = np.zeros(hd)
            want[i] = np.cos(a)
            want[i + hd // 2] = np.sin(a)
            assert np.allclose(got, want, atol=2e-7), (i, pos)
            # the partner e_{i+hd/2} goes to -sin(a) e_i + cos(a) e_{i+hd/2}
            v = np.zeros(hd, np.float32)
            v[i + hd // 2] = 1.0
            got = oracle.rope(v, 1, hd, pos, theta)
            want = np.zeros(hd)
            want[i] = -np.sin(a)
            want[i + hd // 2] = np.cos(a)
            assert np.allclose(got, want, atol=2e-7), (i, pos)


def test_rope_preserves_pair_norms():
    hd = 64
    v = RNG.standard_normal(3 * hd).astype(np.float32)
    r = oracle.rope(v, 3, hd, 777, 500000.0).reshape(3, hd).astype(np.float64)
    v0 = v.reshape(3, hd).astype(np.float64)
    h = hd // 2
    n0 = v0[:, :h] ** 2 + v0[:, h:] ** 2
    n1 = r[:, :h] ** 2 + r[:, h:] ** 2
    assert np.allclose(n0, n1, rtol=1e-6)


def test_rope_scores_depend_only_on_relative_position():
    hd, theta = 64, 10000.0
    q = RNG.standard_normal(hd).astype(np.float32)
    k = RNG.standard_normal(hd).astype(np.float32)

    def score(m, n):
        return float(np.dot(oracle.rope(q, 1, hd, m, theta).astype(np.float64),
                            oracle.rope(k, 1, hd, n, theta).astype(np.float64)))

    base = score(3, 1)
    scale = np.linalg.norm(q) * np.linalg.norm(k)
    for shift in (1, 10, 500):
        assert abs(score(3 + shift, 1 + shift) - base) < 2e-5 * scale
    assert abs(score(5, 1) - base) > 1e-3 * scale  # a different offset does change it


def test_rope_half_split_equals_adjacent_pairs_under_row_permutation():
    # GOTOken, "The rotary convention": HF rotates (j, j+hd/2), llama2.c rotates adjacent
    # pairs; permuting the rows of Wq and Wk maps one onto the other and preserves the
    # attention dot products.
    hd, theta, dim = 16, 10000.0, 32
    wq = RNG.standard_normal((hd, dim)).astype(np.float32)
    wk = RNG.standard_normal((hd, dim)).astype(np.float32)
    x = RNG.standard_normal(dim).astype(np.float32)
    y = RNG.standard_normal(dim).astype(np.float32)
    perm = np.empty(hd, dtype=np.int64)
    perm[0::2] = np.arange(hd // 2)
    perm[1::2] = np.arange(hd // 2) + hd // 2

    def adjacent_rope(v, pos):
        v = v.astype(np.float64).copy()
        for i in range(hd // 2):
            a = pos * theta ** (-2.0 * i / hd)
            c, s = np.cos(a), np.sin(a)
            u, w = v[2 * i], v[2 * i + 1]
            v[2 * i], v[2 * i + 1] = u * c - w * s, u * s + w * c
        return v

    for m, n in ((4, 2), (9, 0), (30, 29)):
        half = np.dot(oracle.rope(oracle.matvec(wq, x), 1, hd, m, theta).astype(np.float64),
                      oracle.rope(oracle.matvec(wk, y), 1, hd, n, theta).astype(np.float64))
        adj = np.dot(adjacent_rope(wq[perm].astype(np.float64) @ x, m),
                     adjacent_rope(wk[perm].astype(np.float64) @ y, n))
        assert abs(half - adj) < 1e-4 * max(1.0, abs(adj))


# ----------------------------------------------------------------------------- attention

def _attn64(q, K, V):
    s = K.astype(np.float64) @ q.astype(np.float64) / np.sqrt(q.size)
    p = np.exp(s - s.max())
    p /= p.sum()
    return p @ V.astype(np.float64), p


def test_attention_brute_force_fp64_tiny():
    for hd in (2, 4, 16):
        for n in range(1, 9):
            q = RNG.standard_normal(hd).astype(np.float32)
            K = RNG.standard_normal((n, hd)).astype(np.float32)
            V = RNG.standard_normal((n, hd)).astype(np.float32)
            got, probs = oracle.attend_probs(q, K, V)
            want, p64 = _attn64(q, K, V)
            assert np.allclose(got, want, rtol=1e-5, atol=1e-5 * np.abs(want).max())
            assert np.allclose(probs, p64, rtol=1e-5, atol=1e-7)


def test_softmax_rows_sum_to_one():
    for n in (1, 2, 17, 261, 1024):
        q = RNG.standard_normal(64).astype(np.float32) * 3
        K = RNG.standard_normal((n, 64)).astype(np.float32)
        V = RNG.standard_normal((n, 64)).astype(np.float32)
        _, p = oracle.attend_probs(q, K, V)
        assert abs(float(np.sum(p, dtype=np.float64)) - 1.0) < 1e-6
        assert np.all(p >= 0)


def test_attention_special_cases():
    hd = 16
    # one cached position: the softmax weight is exactly 1, the output is v exactly
    q = RNG.standard_normal(hd).astype(np.float32)
    K = RNG.standard_normal((1, hd)).astype(np.float32)
    V = RNG.standard_normal((1, hd)).astype(np.float32)
    assert np.array_equal(oracle.attend(q, K, V), V[0])
    # zero query: uniform weights, the output is the mean of V
    n = 7
    K = RNG.standard_normal((n, hd)).astype(np.float32)
    V = RNG.standard_normal((n, hd)).astype(np.float32)
    got = oracle.attend(np.zeros(hd, np.float32), K, V)
    assert np.allclose(got, V.astype(np.float64).mean(0), rtol=1e-6, atol=1e-6)
    # a dominant key: the output is that key's value
    K = np.zeros((n, hd), np.float32)
    K[3] = 100.0
    q = np.ones(hd, np.float32)
    assert np.allclose(oracle.attend(q, K, V), V[3], atol=1e-6)
    # permuting the (key, value) pairs together leaves the output unchanged
    K = RNG.standard_normal((n, hd)).astype(np.float32)
    perm = RNG.permutation(n)
    a = oracle.attend(q, K, V)
    b = oracle.attend(q, K[perm], V[perm])
    assert np.allclose(a, b, rtol=1e-5, atol=1e-6)


# ----------------------------------------------------------------------------- SwiGLU

def test_silu_mul_against_fp64_and_identities():
    a = (RNG.standard_normal(1000) * 4).astype(np.float32)
    b = RNG.standard_normal(1000).astype(np.float32)
    got = oracle.silu_mul(a, b).astype(np.float64)
    a64 = a.astype(np.float64)
    want = a64 / (1 + np.exp(-a64)) * b
    assert np.allclose(got, want, rtol=1e-6, atol=1e-7)
    one = np.ones(5, np.float32)
    z = oracle.silu_mul(np.zeros(5, np.float32), one)
    assert np.all(z == 0)
    big = np.array([30.0, 50.0], np.float32)
    assert np.allclose(oracle.silu_mul(big, np.ones(2, np.float32)), big, rtol=1e-6)
    assert np.all(np.abs(oracle.silu_mul(-big, np.ones(2, np.float32))) < 1e-10)
    # silu(a) - silu(-a) = a
    d = oracle.silu_mul(a, np.ones_like(a)) - oracle.silu_mul(-a, np.ones_like(a))
    assert np.allclose(d, a, rtol=1e-5, atol=1e-6)


# ----------------------------------------------------------------------------- argmax

def test_argmax_lowest_index_on_tie_and_nan_is_an_error():
    x = np.array([1.0, 5.0, 2.0, 5.0, 5.0], np.float32)
    assert oracle.argmax(x) == 1
    assert oracle.argmax(np.zeros(9, np.float32)) == 0
    x = RNG.standard_normal(49152).astype(np.float32)
    assert oracle.argmax(x) == int(np.argmax(x))
    x[17] = np.nan
    assert oracle.argmax(x) == -1


# ----------------------------------------------------------------------------- accounting

def test_parameter_accounting_matches_pages():
    # GOTOken: "SmolLM2-135M has 134.5 million weights" and a 270 MB bf16 checkpoint.
    s = synth.SMOL
    n = synth.n_params(s)
    assert n == 134_515_008
    assert round(n / 1e6, 1) == 134.5
    assert synth.weight_bytes(s) == 269_030_016
    assert abs(synth.weight_bytes(s) / 1e6 - 270) < 1.0
    assert oracle.lib().orc_weight_count(oracle.config_of(s)) == n


def test_kv_cache_size_closed_form():
    # nanochat KV memory example (L=6, B=4, H=6, T=2048, D=64, bf16): 2*L*B*H*T*D*2 bytes
    L, B, H, T, D = 6, 4, 6, 2048, 64
    assert 2 * L * B * H * T * D * 2 == 75_497_472


# ----------------------------------------------------------------------------- model level

def _tiny(**kw):
    return synth.TINY.replace(**kw)


def _model_weights(s, seed=1234):
    return synth.make_weights(s, seed=seed)


def test_cached_equals_uncached_bitwise_and_pass_counts():
    # GOTOken, "About one token per second": 5-token prompt + 8 new tokens took 68
    # uncached forward passes and 12 cached ones, with bit-identical output.
    wl = synth.WORKLOADS["tiny"]
    s = wl.shape
    W = _model_weights(s)
    prompt = synth.make_prompt(s, 0, wl.prompt_len)
    m = oracle.Model(s, W)
    logits, nid = m.prefill(0, prompt)
    cached_ids, cached_logits = [nid], [logits]
    for step in range(wl.decode_steps):
        lg, ids = m.decode_step([0], [cached_ids[-1]], [wl.prompt_len + step])
        cached_ids.append(int(ids[0]))
        cached_logits.append(lg[0])
    assert len(cached_ids) == 8
    assert m.passes == 12

    u = oracle.Model(s, W)
    seq = list(prompt)
    for k in range(8):
        lg, nid = u.forward_uncached(seq)
        assert nid == cached_ids[k]
        assert np.array_equal(lg.view(np.uint32), cached_logits[k].view(np.uint32))
        seq.append(nid)
    assert u.passes == 68


@pytest.mark.parametrize("kw", [dict(kv_dtype=DTYPE_BF16), dict(n_kv_heads=1),
                                dict(n_kv_heads=4), dict(weight_dtype=DTYPE_BF16)])
def test_cached_equals_uncached_variants(kw):
    s = _tiny(**kw)
    W = _model_weights(s)
    prompt = synth.make_prompt(s, 3, 9)
    m = oracle.Model(s, W)
    lg, nid = m.prefill(0, prompt[:4])
    toks = list(prompt[:4])
    for p in range(4, 9):
        lg, ids = m.decode_step([0], [prompt[p]], [p])
        toks.append(prompt[p])
        u = oracle.Model(s, W)
        ul, uid = u.forward_uncached(toks)
        assert np.array_equal(ul.view(np.uint32), lg[0].view(np.uint32))


def _decoder_fp64(s, W, tokens):
    """Brute-force float64 restatement of the decoder over a whole prompt (matrix form,
    causal mask), returning the last position's logits."""
    f = synth.bf16_to_f32(W) if s.weight_dtype == DTYPE_BF16 else W
    f = f.astype(np.float64)
    T = lambda name, l=-1: synth.tensor(f, s, name, l)
    H, KV, hd, dim = s.n_heads, s.n_kv_heads, s.head_dim, s.dim
    E = T("token_emb").reshape(s.vocab, dim)
    X = E[np.asarray(tokens)]
    n = len(tokens)
    pos = np.arange(n)
    half = hd // 2
    freqs = s.rope_theta ** (-2.0 * np.arange(half) / hd)
    ang = pos[:, None] * freqs[None, :]
    cos, sin = np.cos(ang), np.sin(ang)

    def norm(x, g):
        return x / np.sqrt(np.mean(x * x, -1, keepdims=True) + s.norm_eps) * g

    def rope(x):  # [n, heads, hd]
        a, b = x[..., :half], x[..., half:]
        c, sn = cos[:, None, :], sin[:, None, :]
        return np.concatenate([a * c - b * sn, a * sn + b * c], -1)

    mask = np.tril(np.ones((n, n), bool))
    for l in range(s.n_layers):
        xn = norm(X, T("attn_norm", l))
        q = rope((xn @ T("wq", l).reshape(H * hd, dim).T).reshape(n, H, hd))
        k = rope((xn @ T("wk", l).reshape(KV * hd, dim).T).reshape(n, KV, hd))
        v = (xn @ T("wv", l).reshape(KV * hd, dim).T).reshape(n, KV, hd)
        o = np.empty((n, H, hd))
        for h in range(H):
            g = h // (H // KV)
            sc = q[:, h, :] @ k[:, g, :].T / np.sqrt(hd)
            sc = np.where(mask, sc, -np.inf)
            p = np.exp(sc - sc.max(-1, keepdims=True))
            p /= p.sum(-1, keepdims=True)
            o[:, h, :] = p @ v[:, g, :]
        X = X + o.reshape(n, H * hd) @ T("wo", l).reshape(dim, H * hd).T
        xn = norm(X, T("ffn_norm", l))
        a = xn @ T("w1", l).reshape(s.hidden, dim).T
        b = xn @ T("w3", l).reshape(s.hidden, dim).T
        X = X + (a / (1 + np.exp(-a)) * b) @ T("w2", l).reshape(dim, s.hidden).T
    return E @ norm(X[-1], T("output_norm"))


@pytest.mark.parametrize("kw", [dict(), dict(n_kv_heads=1), dict(n_kv_heads=4),
                                dict(weight_dtype=DTYPE_BF16)])
def test_whole_model_against_fp64_brute_force(kw):
    s = _tiny(**kw)
    W = _model_weights(s, seed=99)
    # larger weights so that every block visibly moves the residual stream
    if s.weight_dtype == DTYPE_F32:
        W = W.copy()
        for name, l, off, cnt in synth.layout(s):
            if not name.endswith("norm") and name != "token_emb":
                W[off:off + cnt] *= 10
    prompt = synth.make_prompt(s, 1, 11)
    m = oracle.Model(s, W)
    lg, _ = m.prefill(0, prompt)
    want = _decoder_fp64(s, W, prompt)
    err = np.abs(lg.astype(np.float64) - want).max()
    assert err <= 1e-5 * np.abs(want).max(), err


def test_zero_wo_and_w2_give_embedding_closed_form():
    # With Wo = W2 = 0 both residual updates vanish, so the final stream is the
    # embedding row and logits = E . rmsnorm(E[tok]).
    s = _tiny()
    W = _model_weights(s).copy()
    for name, l, off, cnt in synth.layout(s):
        if name in ("wo", "w2"):
            W[off:off + cnt] = 0
    E = synth.tensor(W, s, "token_emb").reshape(s.vocab, s.dim).astype(np.float64)
    prompt = synth.make_prompt(s, 2, 6)
    m = oracle.Model(s, W)
    lg, nid = m.prefill(0, prompt)
    x = E[prompt[-1]]
    want = E @ (x / np.sqrt(np.mean(x * x) + s.norm_eps))
    assert np.allclose(lg, want, rtol=0, atol=1e-5 * np.abs(want).max())
    assert nid == int(np.argmax(want))


def _repeat_kv_heads(s_gqa, W, s_mha):
    """MHA weights whose kv head j is the GQA model's kv head j // (H/KV)."""
    out = np.empty(synth.n_params(s_mha), dtype=W.dtype)
    group = s_gqa.n_heads // s_gqa.n_kv_heads
    hd, dim = s_gqa.head_dim, s_gqa.dim
    src = {(n, l): (o, c) for n, l, o, c in synth.layout(s_gqa)}
    for name, l, off, cnt in synth.layout(s_mha):
        so, sc = src[(name, l)]
        if name in ("wk", "wv"):
            rows = W[so:so + sc].reshape(s_gqa.n_kv_heads, hd, dim)
            out[off:off + cnt] = np.repeat(rows, group, axis=0).ravel()
        else:
            out[off:off + cnt] = W[so:so + sc]
    return out


@pytest.mark.parametrize("kv", [1, 2])
def test_gqa_equals_mha_with_repeated_kv_heads_bitwise(kv):
    # kasahare "Architecture": GQA accepts n_kv_heads < n_heads, = for MHA, 1 for MQA.
    s_g = _tiny(n_kv_heads=kv)
    s_m = _tiny(n_kv_heads=s_g.n_heads)
    W = _model_weights(s_g, seed=7)
    Wm = _repeat_kv_heads(s_g, W, s_m)
    prompt = synth.make_prompt(s_g, 4, 8)
    a = oracle.Model(s_g, W)
    b = oracle.Model(s_m, Wm)
    la, ia = a.prefill(0, prompt)
    lb, ib = b.prefill(0, prompt)
    assert np.array_equal(la.view(np.uint32), lb.view(np.uint32))
    for p in range(8, 12):
        la, _ = a.decode_step([0], [ia], [p])
        lb, _ = b.decode_step([0], [ia], [p])
        assert np.array_equal(la.view(np.uint32), lb.view(np.uint32))


def test_bf16_cache_rounds_layer0_kv_on_append():
    s32 = _tiny()
    s16 = _tiny(kv_dtype=DTYPE_BF16)
    W = _model_weights(s32)
    prompt = synth.make_prompt(s32, 0, 10)
    a = oracle.Model(s32, W)
    b = oracle.Model(s16, W)
    a.prefill(0, prompt)
    b.prefill(0, prompt)
    ka, va = a.kv(0, 0)
    kb, vb = b.kv(0, 0)
    assert np.array_equal(kb, oracle.bf16_round(ka))
    assert np.array_equal(vb, oracle.bf16_round(va))
    assert np.all(kb.view(np.uint32) & 0xFFFF == 0)


def test_layer0_kv_depends_only_on_token_and_position():
    s = _tiny()
    W = _model_weights(s)
    prompt = synth.make_prompt(s, 5, 12)
    m = oracle.Model(s, W)
    m.prefill(0, prompt)
    K, V = m.kv(0, 0)
    E = synth.tensor(W, s, "token_emb").reshape(s.vocab, s.dim).astype(np.float64)
    wk = synth.tensor(W, s, "wk", 0).reshape(-1, s.dim).astype(np.float64)
    wv = synth.tensor(W, s, "wv", 0).reshape(-1, s.dim).astype(np.float64)
    half = s.head_dim // 2
    for p, tok in enumerate(prompt):
        k1, v1 = m.layer0_kv(int(tok), p)
        assert np.array_equal(k1, K[:, p, :]) and np.array_equal(v1, V[:, p, :])
        x = E[tok]
        xn = x / np.sqrt(np.mean(x * x) + s.norm_eps)
        k = (wk @ xn).reshape(s.n_kv_heads, s.head_dim)
        a = p * s.rope_theta ** (-2.0 * np.arange(half) / s.head_dim)
        k = np.concatenate([k[:, :half] * np.cos(a) - k[:, half:] * np.sin(a),
                            k[:, :half] * np.sin(a) + k[:, half:] * np.cos(a)], 1)
        assert np.allclose(K[:, p, :], k, atol=1e-6)
        assert np.allclose(V[:, p, :], (wv @ xn).reshape(s.n_kv_heads, -1), atol=1e-6)


def test_batch_rows_are_independent_bitwise():
    s = _tiny(max_batch=3)
    W = _model_weights(s)
    prompts = [synth.make_prompt(s, r, 4 + r) for r in range(3)]
    joint = oracle.Model(s, W)
    first = []
    for r in range(3):
        _, nid = joint.prefill(r, prompts[r])
        first.append(nid)
    lj, ij = joint.decode_step([2, 0, 1], [first[2], first[0], first[1]],
                               [len(prompts[2]), len(prompts[0]), len(prompts[1])])
    for i, r in enumerate([2, 0, 1]):
        solo = oracle.Model(s, W)
        solo.prefill(1, prompts[r])
        ls, _ = solo.decode_step([1], [first[r]], [len(prompts[r])])
        assert np.array_equal(ls[0].view(np.uint32), lj[i].view(np.uint32))


def test_api_errors():
    s = _tiny(max_batch=2)
    m = oracle.Model(s, _model_weights(s))
    p = synth.make_prompt(s, 0, 5)
    m.prefill(0, p)
    with pytest.raises(oracle.OracleError) as e:
        m.prefill(0, p)
    assert e.value.code == oracle.ESTATE
    assert m.decode_step_rc([0], [1], [4]) == oracle.EPOS
    assert m.decode_step_rc([0, 0], [1, 1], [5, 5]) == oracle.EINVAL
    assert m.decode_step_rc([0], [s.vocab], [5]) == oracle.EINVAL
    m.reset(0)
    assert m.seq_len(0) == 0
    m.prefill(0, synth.make_prompt(s, 0, s.max_seq))
    assert m.decode_step_rc([0], [1], [s.max_seq]) == oracle.ECAPACITY
    m.reset(-1)
    assert m.seq_len(0) == 0 and m.seq_len(1) == 0
