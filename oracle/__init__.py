"""ctypes wrapper around the fp32 CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py``; never by the CUDA library or its binding.

The shared object is built with plain gcc, ``-O2 -ffp-contract=off`` (no fused
multiply-add, so every product and sum rounds on its own, as in GOTOken's fp32
replay), single-threaded.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_SO = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16, Q8 = 0, 1, 2
Q8_BLOCK = 32
OK, EINVAL, ENOMEM, ECAPACITY, EPOS, ESTATE = 0, -1, -2, -3, -4, -5


def build(force: bool = False) -> str:
    """Compile liboracle.so beside the sources (when missing or stale).

    ``ORACLE_SO`` names a prebuilt variant instead; the mutation test uses it to run
    the pins against copies of the oracle with a planted mistake.
    """
    if os.environ.get("ORACLE_SO"):
        return os.environ["ORACLE_SO"]
    stale = (not os.path.exists(_SO) or
             os.path.getmtime(_SO) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if force or stale:
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("dim", "n_layers", "n_heads", "n_kv_heads", "head_dim", "hidden", "vocab",
                 "max_seq", "max_batch")] + \
               [("rope_theta", ctypes.c_float), ("norm_eps", ctypes.c_float),
                ("weight_dtype", ctypes.c_int32), ("kv_dtype", ctypes.c_int32)]


def config_of(shape) -> Config:
    return Config(shape.dim, shape.n_layers, shape.n_heads, shape.n_kv_heads, shape.head_dim,
                  shape.hidden, shape.vocab, shape.max_seq, shape.max_batch,
                  float(shape.rope_theta), float(shape.norm_eps), int(shape.weight_dtype),
                  int(shape.kv_dtype))


_P = ctypes.c_void_p
_I = ctypes.c_int
_I32 = ctypes.c_int32
_F = ctypes.c_float


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            sig = {
                "orc_bf16_up": (_F, [ctypes.c_uint16]),
                "orc_bf16_round": (_F, [_F]),
                "orc_rmsnorm": (None, [_P, _P, _P, _I, _F]),
                "orc_matvec": (None, [_P, _P, _P, _I, _I]),
                "orc_rope": (None, [_P, _I, _I, _I, _F]),
                "orc_attend": (None, [_P, _P, _P, _P, _I, _I, _P]),
                "orc_silu_mul": (None, [_P, _P, _P, _I]),
                "orc_argmax": (_I32, [_P, _I]),
                "orc_quantize_q8_row": (None, [_P, _I, _P, _P]),
                "orc_weight_count": (ctypes.c_size_t, [ctypes.POINTER(Config)]),
                "orc_create": (_I, [ctypes.POINTER(Config), _P, ctypes.c_size_t, ctypes.POINTER(_P)]),
                "orc_destroy": (None, [_P]),
                "orc_prefill": (_I, [_P, _I32, _P, _I32, _P, _P]),
                "orc_decode_step": (_I, [_P, _I32, _P, _P, _P, _P, _P]),
                "orc_reset": (_I, [_P, _I32]),
                "orc_seq_len": (_I32, [_P, _I32]),
                "orc_passes": (ctypes.c_int64, [_P]),
                "orc_copy_kv": (_I, [_P, _I32, _I32, _P, _P]),
                "orc_layer0_kv": (_I, [_P, _I32, _I32, _P, _P]),
                "orc_forward_uncached": (_I, [_P, _P, _I32, _P, _P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# ------------------------------------------------------------------ scalar pieces

def bf16_up(b: int) -> float:
    return lib().orc_bf16_up(int(b))


def bf16_round(x) -> np.ndarray:
    x = _f32(x)
    f = lib().orc_bf16_round
    return np.array([f(float(v)) for v in x.ravel()], dtype=np.float32).reshape(x.shape)


def rmsnorm(x, g, eps: float) -> np.ndarray:
    x, g = _f32(x), _f32(g)
    out = np.empty_like(x)
    lib().orc_rmsnorm(_ptr(out), _ptr(x), _ptr(g), x.size, eps)
    return out


def matvec(w, x) -> np.ndarray:
    w, x = _f32(w), _f32(x)
    n_out, n_in = w.shape
    out = np.empty(n_out, dtype=np.float32)
    lib().orc_matvec(_ptr(out), _ptr(w), _ptr(x), n_in, n_out)
    return out


def rope(v, n_heads: int, head_dim: int, pos: int, theta: float) -> np.ndarray:
    v = _f32(v).copy()
    lib().orc_rope(_ptr(v), n_heads, head_dim, pos, theta)
    return v


def attend(q, K, V) -> np.ndarray:
    q, K, V = _f32(q), _f32(K), _f32(V)
    n_ctx, hd = K.shape
    out = np.empty(hd, dtype=np.float32)
    scores = np.empty(max(n_ctx, 1), dtype=np.float32)
    lib().orc_attend(_ptr(out), _ptr(q), _ptr(K), _ptr(V), n_ctx, hd, _ptr(scores))
    return out


def attend_probs(q, K, V) -> Tuple[np.ndarray, np.ndarray]:
    """Attention output plus the normalised probabilities the oracle used."""
    q, K, V = _f32(q), _f32(K), _f32(V)
    n_ctx, hd = K.shape
    out = np.empty(hd, dtype=np.float32)
    scores = np.empty(n_ctx, dtype=np.float32)
    lib().orc_attend(_ptr(out), _ptr(q), _ptr(K), _ptr(V), n_ctx, hd, _ptr(scores))
    return out, scores


def silu_mul(a, b) -> np.ndarray:
    a, b = _f32(a), _f32(b)
    h = np.empty_like(a)
    lib().orc_silu_mul(_ptr(h), _ptr(a), _ptr(b), a.size)
    return h


def argmax(x) -> int:
    x = _f32(x)
    return int(lib().orc_argmax(_ptr(x), x.size))


def quantize_q8_row(w) -> Tuple[np.ndarray, np.ndarray]:
    """One weight row to int8 blocks of Q8_BLOCK: (q int8[n], d float32[ceil(n / 32)])."""
    w = _f32(w).ravel()
    n = w.size
    q = np.zeros(n, dtype=np.int8)
    d = np.zeros((n + Q8_BLOCK - 1) // Q8_BLOCK, dtype=np.float32)
    lib().orc_quantize_q8_row(_ptr(w), n, _ptr(q), _ptr(d))
    return q, d


# ------------------------------------------------------------------ the model

class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what} failed with oracle status {code}")
        self.code = code


class Model:
    """One oracle instance: weights (canonical buffer) + its own KV cache."""

    def __init__(self, shape, weights: np.ndarray):
        self.shape = shape
        self.cfg = config_of(shape)
        w = np.ascontiguousarray(weights)
        h = ctypes.c_void_p()
        rc = lib().orc_create(ctypes.byref(self.cfg), _ptr(w), w.nbytes, ctypes.byref(h))
        if rc != OK:
            raise OracleError(rc, "orc_create")
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            lib().orc_destroy(self._h)
            self._h = None

    __del__ = close

    def _check(self, rc: int, what: str):
        if rc != OK:
            raise OracleError(rc, what)

    def prefill(self, seq: int, tokens) -> Tuple[np.ndarray, int]:
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        logits = np.empty(self.shape.vocab, dtype=np.float32)
        nid = ctypes.c_int32()
        self._check(lib().orc_prefill(self._h, seq, _ptr(t), t.size, _ptr(logits),
                                      ctypes.byref(nid)), "orc_prefill")
        return logits, int(nid.value)

    def decode_step(self, seq_ids, tokens, positions) -> Tuple[np.ndarray, np.ndarray]:
        s = np.ascontiguousarray(seq_ids, dtype=np.int32)
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        p = np.ascontiguousarray(positions, dtype=np.int32)
        logits = np.empty((s.size, self.shape.vocab), dtype=np.float32)
        ids = np.empty(s.size, dtype=np.int32)
        self._check(lib().orc_decode_step(self._h, s.size, _ptr(s), _ptr(t), _ptr(p),
                                          _ptr(logits), _ptr(ids)), "orc_decode_step")
        return logits, ids

    def decode_step_rc(self, seq_ids, tokens, positions) -> int:
        s = np.ascontiguousarray(seq_ids, dtype=np.int32)
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        p = np.ascontiguousarray(positions, dtype=np.int32)
        return lib().orc_decode_step(self._h, s.size, _ptr(s), _ptr(t), _ptr(p), None, None)

    def reset(self, seq: int = -1):
        self._check(lib().orc_reset(self._h, seq), "orc_reset")

    def seq_len(self, seq: int) -> int:
        return int(lib().orc_seq_len(self._h, seq))

    @property
    def passes(self) -> int:
        return int(lib().orc_passes(self._h))

    def kv(self, layer: int, seq: int) -> Tuple[np.ndarray, np.ndarray]:
        """Cached K and V of one (layer, sequence): arrays [kv_heads][len][head_dim]."""
        n = self.seq_len(seq)
        s = self.shape
        k = np.empty((s.n_kv_heads, n, s.head_dim), dtype=np.float32)
        v = np.empty_like(k)
        rc = lib().orc_copy_kv(self._h, layer, seq, _ptr(k), _ptr(v))
        if rc < 0:
            raise OracleError(rc, "orc_copy_kv")
        return k, v

    def layer0_kv(self, tok: int, pos: int) -> Tuple[np.ndarray, np.ndarray]:
        s = self.shape
        k = np.empty(s.n_kv_heads * s.head_dim, dtype=np.float32)
        v = np.empty_like(k)
        self._check(lib().orc_layer0_kv(self._h, tok, pos, _ptr(k), _ptr(v)), "orc_layer0_kv")
        return k.reshape(s.n_kv_heads, s.head_dim), v.reshape(s.n_kv_heads, s.head_dim)

    def forward_uncached(self, tokens) -> Tuple[np.ndarray, int]:
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        logits = np.empty(self.shape.vocab, dtype=np.float32)
        nid = ctypes.c_int32()
        self._check(lib().orc_forward_uncached(self._h, _ptr(t), t.size, _ptr(logits),
                                               ctypes.byref(nid)), "orc_forward_uncached")
        return logits, int(nid.value)


def greedy_run(shape, weights, prompts, steps: int, rows: Optional[list] = None):
    """Prefill each row's prompt, then ``steps`` batched greedy decode steps.

    Returns ``(ids, logits)``: ``ids[r]`` is the list of generated ids (the prefill
    argmax first, then one per step) and ``logits[r]`` a list of fp32 logit vectors
    (prefill last position first).  Each row runs as its own sequence id.
    """
    rows = list(range(len(prompts))) if rows is None else rows
    m = Model(shape, weights)
    ids = {r: [] for r in rows}
    logs = {r: [] for r in rows}
    for i, r in enumerate(rows):
        lg, nid = m.prefill(i, prompts[r])
        ids[r].append(nid)
        logs[r].append(lg)
    for step in range(steps):
        seqs = list(range(len(rows)))
        toks = [ids[r][-1] for r in rows]
        poss = [len(prompts[r]) + step for r in rows]
        lg, nid = m.decode_step(seqs, toks, poss)
        for i, r in enumerate(rows):
            ids[r].append(int(nid[i]))
            logs[r].append(lg[i])
    m.close()
    return ids, logs
