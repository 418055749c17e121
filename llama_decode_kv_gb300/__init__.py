"""Thin Python binding of the GB300 decode library (``libslm.so``, C ABI in
``include/slm.h``).

Argument marshalling only: every step of the decode path runs in the library's CUDA
kernels.  PyTorch provides device memory and streams.  Importing this package without
the built library raises ``ImportError``: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libslm.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "slm.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python llama_decode_kv_gb300/build.py` "
        "(CUDA toolkit required); there is no CPU fallback")

_lib = ctypes.CDLL(LIB_PATH)

SLM_F32, SLM_BF16 = 0, 1
STATUS = {0: "SLM_OK", -1: "SLM_EINVAL", -2: "SLM_ENOMEM", -3: "SLM_ECAPACITY", -4: "SLM_EPOS",
          -5: "SLM_ESTATE", -6: "SLM_ECUDA", -7: "SLM_ETIMEOUT", -8: "SLM_EDEVICE",
          -9: "SLM_EUNSUPPORTED"}
for _code, _name in STATUS.items():
    globals()[_name] = _code


class slm_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("dim", "n_layers", "n_heads", "n_kv_heads", "head_dim", "hidden", "vocab",
                 "max_seq", "max_batch")] + \
               [("rope_theta", ctypes.c_float), ("norm_eps", ctypes.c_float),
                ("weight_dtype", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
                ("kv_page_size", ctypes.c_int32), ("kv_pages", ctypes.c_int32)]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_SIGS = {
    "slm_create": (ctypes.c_int, [ctypes.POINTER(slm_config), _P, ctypes.c_size_t, ctypes.POINTER(_P)]),
    "slm_prefill": (ctypes.c_int, [_P, _I32, _P, _I32, _P, _P, _P]),
    "slm_decode_step": (ctypes.c_int, [_P, _I32, _P, _P, _P, _P, _P, _P]),
    "slm_reset": (ctypes.c_int, [_P, _I32]),
    "slm_seq_len": (_I32, [_P, _I32]),
    "slm_kv_pages_free": (_I32, [_P]),
    "slm_quantize_q8": (ctypes.c_int, [_P, _I32, _I32, _P, _P]),
    "slm_debug_page_table": (_I32, [_P, _I32, _P, _I32]),
    "slm_fork": (ctypes.c_int, [_P, _I32, _I32, _P, _P]),
    "slm_prefill_batch": (ctypes.c_int, [_P, _I32, _P, _P, _P, _P, _P, _P]),
    "slm_sample": (ctypes.c_int, [_I32, _I32, _P, _I32, ctypes.c_float, _I32, ctypes.c_float, _P, _P, _P]),
    "slm_sync": (ctypes.c_int, [_P, _P]),
    "slm_destroy": (None, [_P]),
    "slm_last_error": (ctypes.c_char_p, [_P]),
    "slm_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "slm_debug_copy_kv": (ctypes.c_int, [_P, _I32, _I32, _I32, _P, _P]),
    "slm_debug_fill_kv": (ctypes.c_int, [_P, ctypes.c_float]),
    "slm_debug_trace": (ctypes.c_int, [_P, _I32, _P, ctypes.c_size_t]),
    "slm_debug_plan": (ctypes.c_int, [ctypes.POINTER(slm_config), _I32, _P, _I32]),
    "slm_debug_cluster": (ctypes.c_int, [_P, _P, _I32]),
    "slm_debug_faults": (ctypes.c_int, [_P, ctypes.c_ulonglong, _I32]),
    "slm_debug_gemm_bf16": (ctypes.c_int, [_I32, _I32, _I32, _P, _P, _P, _P]),
    "slm_attention_workspace_bytes": (ctypes.c_size_t, [_I32, _I32, _I32, _I32]),
    "slm_attention_decode": (ctypes.c_int, [_I32, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P,
                                            _P, ctypes.c_size_t, _P]),
    "slm_attention_noalloc_max_bytes": (ctypes.c_size_t, []),
    "slm_attention_decode_noalloc": (ctypes.c_int, [_I32, _I32, _I32, _I32, _I32, _I32, _P, _P, _P,
                                                    _P, _P, _P]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args
    globals()[_name] = _fn


def header_symbols(path: str = HEADER) -> list:
    """Every entry point the public header declares."""
    text = open(path).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(slm_\w+)\s*\(", text, re.M)))


class SlmError(RuntimeError):
    def __init__(self, code: int, what: str, detail: str = ""):
        super().__init__(f"{what}: {STATUS.get(code, code)} {detail}".strip())
        self.code = code


def config_from_shape(shape, kv_page_size: int = 0, kv_pages: int = 0) -> slm_config:
    return slm_config(shape.dim, shape.n_layers, shape.n_heads, shape.n_kv_heads, shape.head_dim,
                      shape.hidden, shape.vocab, shape.max_seq, shape.max_batch,
                      float(shape.rope_theta), float(shape.norm_eps), int(shape.weight_dtype),
                      int(shape.kv_dtype), int(kv_page_size), int(kv_pages))


def _ptr(x) -> Optional[int]:
    """Address of a torch tensor or numpy array (None stays None)."""
    if x is None:
        return None
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    return x.data_ptr()


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def attention_decode(q, k_cache, v_cache, ctx_len, out, workspace, kv_dtype: int, stream=None) -> int:
    """slm_attention_decode over torch tensors: q/out [B][H][hd] fp32, caches
    [B][KV][cap][hd], ctx_len a sequence of ints, workspace a uint8 device tensor."""
    B, H, hd = q.shape
    KV, cap = k_cache.shape[1], k_cache.shape[2]
    lens = (ctypes.c_int32 * B)(*[int(x) for x in ctx_len])
    return slm_attention_decode(B, H, KV, hd, cap, kv_dtype, _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                lens, _ptr(out), _ptr(workspace), workspace.numel(),
                                _stream_ptr(stream))


def attention_decode_noalloc(q, k_cache, v_cache, ctx_len, out, kv_dtype: int, stream=None) -> int:
    """slm_attention_decode_noalloc over torch tensors (no workspace argument)."""
    B, H, hd = q.shape
    KV, cap = k_cache.shape[1], k_cache.shape[2]
    lens = (ctypes.c_int32 * B)(*[int(x) for x in ctx_len])
    return slm_attention_decode_noalloc(B, H, KV, hd, cap, kv_dtype, _ptr(q), _ptr(k_cache),
                                        _ptr(v_cache), lens, _ptr(out), _stream_ptr(stream))


def sample(logits, temperature: float, top_k: int, top_p: float, uniforms, next_ids, stream=None) -> int:
    """slm_sample on device tensors: logits [batch][ld] float32, uniforms [batch] float32,
    next_ids [batch] int32.  Returns the status code."""
    batch, ld = int(logits.shape[0]), int(logits.shape[1])
    return slm_sample(batch, ld, _ptr(logits), ld, float(temperature), int(top_k), float(top_p), _ptr(uniforms),
                      _ptr(next_ids), _stream_ptr(stream))


def quantize_q8(w: np.ndarray):
    """slm_quantize_q8 on a [rows][cols] fp32 array: (q int8[rows][cols], d float32[rows][ceil(cols/32)])."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    if w.ndim == 1:
        w = w[None, :]
    rows, cols = w.shape
    q = np.zeros((rows, cols), dtype=np.int8)
    d = np.zeros((rows, (cols + 31) // 32), dtype=np.float32)
    rc = slm_quantize_q8(w.ctypes.data, rows, cols, q.ctypes.data, d.ctypes.data)
    if rc != 0:
        raise SlmError(rc, "slm_quantize_q8")
    return q, d


def plan(shape, sms: int = 152) -> dict:
    """slm_debug_plan: the engine layout for a shape, computed on the host (no GPU)."""
    cfg = config_from_shape(shape)
    out = np.zeros(47, dtype=np.int32)
    rc = slm_debug_plan(ctypes.byref(cfg), sms, out.ctypes.data, out.size)
    if rc != 0:
        raise SlmError(rc, "slm_debug_plan", slm_last_error(None).decode())
    v = [int(x) for x in out]
    d = {"grid": v[0], "roles": v[1], "role0": v[2:7], "own_ld": v[7], "acc_bytes": v[8], "xs_bytes": v[9],
         "ring_slots": v[10], "smem": v[11]}
    for i, name in enumerate(("emb", "qkv", "wo", "w13", "w2")):
        r = v[12 + 7 * i: 19 + 7 * i]
        d[name] = dict(zip(("rows", "K", "KB", "KBp", "nkt", "rows_per_unit", "rows_per_chunk"), r))
    return d


class Engine:
    """One decode context: device weights, KV cache and per-sequence lengths."""

    def __init__(self, shape, weights, kv_page_size: int = 0, kv_pages: int = 0):
        """kv_page_size > 0: a paged KV cache of kv_pages pages (0: enough for every slot)."""
        import torch  # device memory and streams
        self.torch = torch
        self.shape = shape
        self.cfg = config_from_shape(shape, kv_page_size, kv_pages)
        buf = weights if not isinstance(weights, np.ndarray) else np.ascontiguousarray(weights)
        nbytes = buf.nbytes if isinstance(buf, np.ndarray) else buf.numel() * buf.element_size()
        h = ctypes.c_void_p()
        rc = slm_create(ctypes.byref(self.cfg), _ptr(buf), nbytes, ctypes.byref(h))
        if rc != 0:
            raise SlmError(rc, "slm_create", slm_last_error(None).decode())
        self.ctx = h

    def close(self):
        if getattr(self, "ctx", None):
            slm_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, rc: int, what: str):
        if rc != 0:
            raise SlmError(rc, what, slm_last_error(self.ctx).decode())

    # ---------------------------------------------------------------- calls
    def prefill(self, seq: int, tokens, last_logits=None, next_id=None, stream=None) -> int:
        """tokens / last_logits / next_id: torch tensors (device or host) or numpy arrays."""
        n = int(tokens.numel() if hasattr(tokens, "numel") else len(tokens))
        return slm_prefill(self.ctx, seq, _ptr(tokens), n, _ptr(last_logits), _ptr(next_id),
                           _stream_ptr(stream))

    def decode_step(self, seq_ids: Sequence[int], tokens, positions: Sequence[int], logits=None,
                    next_ids=None, stream=None) -> int:
        b = len(seq_ids)
        s = (ctypes.c_int32 * b)(*seq_ids)
        p = (ctypes.c_int32 * b)(*positions)
        return slm_decode_step(self.ctx, b, s, _ptr(tokens), p, _ptr(logits), _ptr(next_ids),
                               _stream_ptr(stream))

    def reset(self, seq: int = -1):
        self._check(slm_reset(self.ctx, seq), "slm_reset")

    def prefill_batch(self, seqs: Sequence[int], tokens, lens: Sequence[int], last_logits=None, next_ids=None,
                      stream=None) -> int:
        """slm_prefill_batch: tokens = device int32 prompts concatenated in seqs order."""
        n = len(seqs)
        sq = (ctypes.c_int32 * n)(*seqs)
        ln = (ctypes.c_int32 * n)(*[int(x) for x in lens])
        return slm_prefill_batch(self.ctx, n, sq, ln, _ptr(tokens), _ptr(last_logits), _ptr(next_ids),
                                 _stream_ptr(stream))

    def fork(self, src: int, dst_seqs: Sequence[int], stream=None) -> int:
        """Clone sequence src's cache into the empty sequences dst_seqs (status code)."""
        d = (ctypes.c_int32 * len(dst_seqs))(*dst_seqs)
        return slm_fork(self.ctx, src, len(dst_seqs), d, _stream_ptr(stream))

    def seq_len(self, seq: int) -> int:
        return int(slm_seq_len(self.ctx, seq))

    def pages_free(self) -> int:
        """slm_kv_pages_free: pages of a paged cache that no sequence holds."""
        n = int(slm_kv_pages_free(self.ctx))
        if n < 0:
            raise SlmError(n, "slm_kv_pages_free", self.last_error())
        return n

    def page_table(self, seq: int) -> np.ndarray:
        """slm_debug_page_table: the page ids of sequence seq (-1: none)."""
        n = int(slm_debug_page_table(self.ctx, seq, None, 0))
        if n < 0:
            raise SlmError(n, "slm_debug_page_table", self.last_error())
        out = np.zeros(n, dtype=np.int32)
        slm_debug_page_table(self.ctx, seq, out.ctypes.data, n)
        return out

    def sync(self, stream=None) -> int:
        return slm_sync(self.ctx, _stream_ptr(stream))

    def last_error(self) -> str:
        return slm_last_error(self.ctx).decode()

    def kv(self, layer: int, seq: int, n_pos: int = -1) -> Tuple[np.ndarray, np.ndarray]:
        n = self.seq_len(seq) if n_pos < 0 else n_pos
        s = self.shape
        k = np.empty((s.n_kv_heads, n, s.head_dim), dtype=np.float32)
        v = np.empty_like(k)
        rc = slm_debug_copy_kv(self.ctx, layer, seq, n, k.ctypes.data, v.ctypes.data)
        if rc < 0:
            raise SlmError(rc, "slm_debug_copy_kv", self.last_error())
        return k, v

    def debug_faults(self, wait_ns: int = 0, lost_publish: int = 0):
        """Shorten the device-side wait limit (0: default) and/or make one publish go
        missing in the following steps (slm_debug_faults)."""
        self._check(slm_debug_faults(self.ctx, int(wait_ns), int(lost_publish)), "slm_debug_faults")

    def cluster_plan(self):
        """None when single-row steps run on the persistent kernel, else a dict of the
        cluster kernel's plan (slm_debug_cluster)."""
        out = np.zeros(12, dtype=np.int32)
        rc = slm_debug_cluster(self.ctx, out.ctypes.data, out.size)
        if rc < 0:
            raise SlmError(rc, "slm_debug_cluster", self.last_error())
        if rc == 0:
            return None
        keys = ("C", "NA", "NF", "grid", "hpc", "ring_slots", "smem", "upc_qkv", "upc_wo", "upc_w13",
                "upc_w2", "upc_emb")
        return dict(zip(keys, (int(v) for v in out)))

    def trace(self, enable: bool = True, fetch: bool = False):
        """Turn the phase timeline on/off; with fetch, return the last step's record as
        uint64 [grid][5 * n_layers + 2][3] (entered, inputs ready, done) in ns."""
        if not fetch:
            rc = slm_debug_trace(self.ctx, int(enable), None, 0)
            if rc < 0:
                raise SlmError(rc, "slm_debug_trace", self.last_error())
            return None
        grid = slm_debug_trace(self.ctx, int(enable), None, 0)
        if grid < 0:
            raise SlmError(grid, "slm_debug_trace", self.last_error())
        out = np.zeros((grid, 5 * self.shape.n_layers + 2, 3), dtype=np.uint64)
        rc = slm_debug_trace(self.ctx, int(enable), out.ctypes.data, out.size)
        if rc < 0:
            raise SlmError(rc, "slm_debug_trace", self.last_error())
        return out

    def fill_kv(self, value: float):
        self._check(slm_debug_fill_kv(self.ctx, float(value)), "slm_debug_fill_kv")

    # ---------------------------------------------------------------- conveniences
    def prefill_checked(self, seq: int, tokens, want_logits: bool = True):
        """Prefill from device tensors; returns (logits or None, next id tensor)."""
        torch = self.torch
        dev = torch.device("cuda")
        t = torch.as_tensor(np.asarray(tokens, dtype=np.int32)).to(dev)
        lg = torch.empty(self.shape.vocab, dtype=torch.float32, device=dev) if want_logits else None
        nid = torch.empty(1, dtype=torch.int32, device=dev)
        self._check(self.prefill(seq, t, lg, nid), "slm_prefill")
        return lg, nid

    def decode_checked(self, seq_ids, tokens_dev, positions, want_logits: bool = True):
        torch = self.torch
        dev = torch.device("cuda")
        b = len(seq_ids)
        lg = torch.empty((b, self.shape.vocab), dtype=torch.float32, device=dev) if want_logits else None
        ids = torch.empty(b, dtype=torch.int32, device=dev)
        self._check(self.decode_step(seq_ids, tokens_dev, positions, lg, ids), "slm_decode_step")
        return lg, ids
