"""C-ABI checks that need no GPU: the library loads, exports every entry point the
public header declares, and rejects bad arguments before touching the device."""
import ctypes

import numpy as np
import pytest

import synth

slm = pytest.importorskip("llama_decode_kv_gb300", reason="libslm.so not built")


def test_library_exports_every_header_symbol():
    names = slm.header_symbols()
    assert {"slm_create", "slm_prefill", "slm_decode_step", "slm_reset", "slm_destroy",
            "slm_sync", "slm_last_error"} <= set(names)
    for n in names:
        assert hasattr(slm._lib, n), f"{n} declared in include/slm.h but not exported"


def test_status_strings():
    for code in slm.STATUS:
        assert slm.slm_status_string(code)
    assert slm.slm_status_string(0) == b"ok"


def _create(cfg, nbytes=None, weights=True):
    buf = np.zeros(max(1, nbytes or 1), dtype=np.uint8)
    h = ctypes.c_void_p()
    rc = slm.slm_create(ctypes.byref(cfg) if cfg is not None else None,
                        buf.ctypes.data if weights else None,
                        buf.nbytes if nbytes is None else nbytes, ctypes.byref(h))
    return rc, h


def _cfg(**kw):
    return slm.config_from_shape(synth.TINY.replace(**kw))


@pytest.mark.parametrize("kw,why", [
    (dict(n_kv_heads=3), "multiple"),
    (dict(dim=66), "dim 66"),
    (dict(head_dim=12), "head_dim"),
    (dict(head_dim=0), "positive"),
    (dict(max_batch=17), "max_batch"),
    (dict(weight_dtype=7), "weight_dtype"),
    (dict(kv_dtype=3), "kv_dtype"),
    (dict(rope_theta=0.0), "rope_theta"),
    (dict(norm_eps=-1.0), "norm_eps"),
])
def test_create_rejects_bad_config_before_any_device_work(kw, why):
    rc, h = _create(_cfg(**kw), nbytes=16)
    assert rc == slm.SLM_EINVAL
    assert not h.value
    assert why in slm.slm_last_error(None).decode()


def test_create_rejects_wrong_size_and_null():
    cfg = _cfg()
    n = synth.n_params(synth.TINY) * 4
    rc, _ = _create(cfg, nbytes=n - 4)
    assert rc == slm.SLM_EINVAL and b"bytes" in slm.slm_last_error(None)
    rc, _ = _create(None, nbytes=n)
    assert rc == slm.SLM_EINVAL
    rc, _ = _create(cfg, nbytes=n, weights=False)
    assert rc == slm.SLM_EINVAL
    assert slm.slm_create(ctypes.byref(cfg), None, 0, None) == slm.SLM_EINVAL


def test_null_context_calls_fail_cleanly():
    assert slm.slm_reset(None, 0) == slm.SLM_EINVAL
    assert slm.slm_seq_len(None, 0) == slm.SLM_EINVAL
    assert slm.slm_sync(None, None) == slm.SLM_EINVAL
    assert slm.slm_prefill(None, 0, None, 1, None, None, None) == slm.SLM_EINVAL
    assert slm.slm_decode_step(None, 1, None, None, None, None, None, None) == slm.SLM_EINVAL
    slm.slm_destroy(None)
