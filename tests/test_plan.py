"""The engine's host-side plan (work split, K tiling, shared-memory layout) for every
workload shape, computed on the CPU through slm_debug_plan: the invariants the decode
kernel relies on, checked without a GPU."""
import math

import pytest

import synth

slm = pytest.importorskip("llama_decode_kv_gb300")

SMEM_LIMIT = 227 * 1024
CHUNK = 8192
MATS = ("emb", "qkv", "wo", "w13", "w2")


def _shapes():
    out = dict((n, wl.shape.replace(max_batch=wl.batch) if wl.batch > wl.shape.max_batch else wl.shape)
               for n, wl in synth.WORKLOADS.items())
    out["smol_b8_f32"] = synth.SMOL.replace(max_batch=8, weight_dtype=synth.DTYPE_F32)
    out["llama_b4"] = synth.LLAMA1B.replace(max_batch=4)
    # block-quantised int8 weights
    out["smol_b1_q8"] = synth.SMOL.replace(weight_dtype=synth.DTYPE_Q8)
    out["smol_b16_q8"] = synth.SMOL.replace(max_batch=16, weight_dtype=synth.DTYPE_Q8, kv_dtype=synth.DTYPE_BF16)
    out["llama_b1_q8"] = synth.LLAMA1B.replace(max_batch=1, weight_dtype=synth.DTYPE_Q8)
    out["llama_b8_q8"] = synth.LLAMA1B.replace(weight_dtype=synth.DTYPE_Q8)
    out["tiny_ragged_q8"] = synth.TINY.replace(max_batch=3, weight_dtype=synth.DTYPE_Q8, dim=72, n_heads=3,
                                               n_kv_heads=1, head_dim=24, hidden=100, vocab=333)
    return out


def _rowbytes(s, KBp):
    """Stored bytes of one row of one K tile: int8 rows carry one fp32 scale per 32."""
    if s.weight_dtype == synth.DTYPE_Q8:
        return KBp + KBp // 32 * 4
    return KBp * (2 if s.weight_dtype == synth.DTYPE_BF16 else 4)


@pytest.mark.parametrize("name", sorted(_shapes()))
@pytest.mark.parametrize("sms", [132, 148, 152])
def test_plan_invariants(name, sms):
    s = _shapes()[name]
    p = slm.plan(s, sms)
    B, esz = s.max_batch, 2 if s.weight_dtype == synth.DTYPE_BF16 else 4
    assert p["grid"] == sms
    assert p["smem"] <= SMEM_LIMIT
    assert p["ring_slots"] % 8 == 0 and 16 <= p["ring_slots"] <= 32
    assert p["smem"] - p["ring_slots"] * CHUNK >= p["xs_bytes"]
    pad = 16 if (B > 8 and esz == 2) else 0  # the batch-16 tensor-core ring pads every row
    for mname in MATS:
        M = p[mname]
        assert M["nkt"] * M["KB"] >= M["K"] > (M["nkt"] - 1) * M["KB"], mname
        assert M["KBp"] % 64 == 0 and M["KBp"] >= M["KB"], mname
        assert M["rows_per_chunk"] % M["rows_per_unit"] == 0 and M["rows_per_chunk"] <= 8, mname
        assert M["rows_per_chunk"] * (_rowbytes(s, M["KBp"]) + pad) <= CHUNK, mname
        # every row starts on a 16-byte boundary (the ring's bulk copies need it)
        assert _rowbytes(s, M["KBp"]) % 16 == 0, mname
        tile = 16 * (M["KBp"] + 8) * 4 if B > 8 else B * M["KBp"] * 4
        extra = s.dim * 4 if mname in ("emb", "qkv", "w13") else 0
        assert tile + extra <= p["xs_bytes"], mname
    for mname in ("emb", "qkv", "w13"):  # the normalised inputs are staged whole
        assert p[mname]["nkt"] == 1, mname
    assert (p["acc_bytes"] > 0) == (p["wo"]["nkt"] > 1 or p["w2"]["nkt"] > 1)
    assert p["qkv"]["rows"] == (s.n_heads + 2 * s.n_kv_heads) * s.head_dim
    assert p["w13"]["rows"] == 2 * s.hidden and p["w13"]["rows_per_unit"] == 2
    if p["roles"]:
        r = p["role0"]
        assert B <= 4 and r[0] == 0 and r[4] == sms and r[2] - r[1] == 16
        assert all(r[i] < r[i + 1] for i in range(4))
        assert p["own_ld"] == math.ceil(s.dim / (r[3] - r[2]))
    else:
        assert p["own_ld"] == math.ceil(s.dim / (sms - sms // 4))


def test_roles_only_for_small_models_at_small_batches():
    plans = {n: slm.plan(s) for n, s in _shapes().items()}
    assert plans["smol_b1"]["roles"] and plans["tiny"]["roles"]
    for n in ("smol_b16", "llama1b_b1", "llama1b_b8", "llama1b_long"):
        assert not plans[n]["roles"], n


def test_smol_batch16_w2_is_one_k_tile_beside_a_16_slot_ring():
    p = slm.plan(synth.WORKLOADS["smol_b16"].shape)
    assert p["w2"]["nkt"] == 1 and p["ring_slots"] == 16 and p["smem"] == SMEM_LIMIT


def test_shapes_that_do_not_fit_are_refused():
    # engines of more than 8 rows stage the normalised input of 16 padded rows whole as
    # bf16 hi + lo planes: dim 2048 needs 131 KB beside a 16-slot ring (98 KB free)
    with pytest.raises(slm.SlmError, match="does not fit"):
        slm.plan(synth.LLAMA1B.replace(max_batch=16))
    with pytest.raises(slm.SlmError):
        slm.plan(synth.LLAMA1B.replace(dim=32768, n_heads=256, n_kv_heads=64, hidden=65536))
    with pytest.raises(slm.SlmError):
        slm.plan(synth.TINY.replace(n_kv_heads=3))  # heads not a multiple of kv heads


@pytest.mark.parametrize("bad", [
    dict(kv_page_size=8),            # below 16 positions
    dict(kv_page_size=48),           # not a power of two
    dict(kv_page_size=0, kv_pages=4),  # a pool without pages
    dict(kv_page_size=16, kv_pages=3),  # cannot hold one max_seq sequence (64 / 16 = 4 pages)
    dict(kv_page_size=16, kv_pages=-1),
    dict(weight_dtype=3),            # no such weight type
])
def test_bad_cache_and_weight_configs_are_refused(bad):
    cfg = slm.config_from_shape(synth.TINY)
    for k, v in bad.items():
        setattr(cfg, k, v)
    import ctypes
    import numpy as np
    out = np.zeros(64, dtype=np.int32)
    rc = slm.slm_debug_plan(ctypes.byref(cfg), 152, out.ctypes.data, out.size)
    assert rc == slm.SLM_EINVAL, (bad, rc)


@pytest.mark.parametrize("good", [dict(kv_page_size=16), dict(kv_page_size=16, kv_pages=4),
                                  dict(kv_page_size=1 << 20), dict(weight_dtype=2)])
def test_paged_and_int8_configs_plan(good):
    cfg = slm.config_from_shape(synth.TINY)
    for k, v in good.items():
        setattr(cfg, k, v)
    import ctypes
    import numpy as np
    out = np.zeros(64, dtype=np.int32)
    assert slm.slm_debug_plan(ctypes.byref(cfg), 152, out.ctypes.data, out.size) == 0
