"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the benchmark.

This module only *makes inputs*: model shapes, random-init weight buffers in the
canonical on-disk order, and random prompt token ids.  It holds none of the
decoder's arithmetic, so both sides of every parity check (the CPU oracle and the
CUDA library) consume byte-identical inputs without sharing any computation.

Canonical weight order (kasahare 0.4.0 / simple-llm, section "On-disk model format
(.sllm)"): ``token_emb[vocab*dim]``; per block ``attn_norm[dim], wq[H*hd*dim],
wk[KV*hd*dim], wv[KV*hd*dim], wo[dim*H*hd], ffn_norm[dim], w1[hidden*dim],
w3[hidden*dim], w2[dim*hidden]``; then ``output_norm[dim]``.  Every matrix is
row-major ``[out][in]`` (GOTOken, "About one token per second": ``W(d, n)`` stored
row-major).  The embedding is tied: it is also the output projection (kasahare,
"Optimisations").

Recipe (the pages only say "random weights, deterministic per --seed", kasahare
"Quick start"):

* one ``numpy.random.default_rng(seed)`` stream (seed 1234), drawn tensor by tensor
  in the canonical order, ``standard_normal(n, float32) * float32(0.02)``;
* RMSNorm gains are exactly 1.0 and consume no draws;
* bf16 weight buffers are the fp32 draws rounded to nearest-even bf16 (bf16 is the
  top half of an fp32 word: GOTOken, "Loading the model and tokenizer");
* prompts: ``default_rng(5678 + row).integers(0, vocab, n, int32)``.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Dict, List, Tuple

import numpy as np

DTYPE_F32 = 0
DTYPE_BF16 = 1
DTYPE_Q8 = 2  # block-quantised int8 weights: the input buffer is fp32, quantised by the consumer

WEIGHT_SEED = 1234
PROMPT_SEED = 5678


@dataclasses.dataclass(frozen=True)
class Shape:
    """Decoder shape plus storage types. Field names follow the C config struct."""

    dim: int
    n_layers: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    hidden: int
    vocab: int
    max_seq: int
    max_batch: int
    rope_theta: float
    norm_eps: float = 1e-5
    weight_dtype: int = DTYPE_BF16
    kv_dtype: int = DTYPE_F32

    def replace(self, **kw) -> "Shape":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class Workload:
    """A named decode workload: a shape, a batch, a prompt length and a step count."""

    name: str
    shape: Shape
    batch: int
    prompt_len: int
    decode_steps: int
    note: str = ""


TINY = Shape(dim=64, n_layers=2, n_heads=4, n_kv_heads=2, head_dim=16, hidden=172,
             vocab=256, max_seq=64, max_batch=1, rope_theta=10000.0,
             weight_dtype=DTYPE_F32, kv_dtype=DTYPE_F32)
SMOL = Shape(dim=576, n_layers=30, n_heads=9, n_kv_heads=3, head_dim=64, hidden=1536,
             vocab=49152, max_seq=1024, max_batch=1, rope_theta=100000.0,
             weight_dtype=DTYPE_BF16, kv_dtype=DTYPE_F32)
LLAMA1B = Shape(dim=2048, n_layers=16, n_heads=32, n_kv_heads=8, head_dim=64,
                hidden=8192, vocab=128256, max_seq=2304, max_batch=8,
                rope_theta=500000.0, weight_dtype=DTYPE_BF16, kv_dtype=DTYPE_BF16)

LONG_2L = LLAMA1B.replace(n_layers=2, hidden=512, vocab=2048, max_batch=4, max_seq=32832)

# The five workloads (plus a reduced long-context one the oracle can finish).  Step counting: a prompt of P tokens is prefilled, its argmax is
# the first generated token, and every further token costs one decode step.
WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", TINY, batch=1, prompt_len=5, decode_steps=7,
                     note="5-token prompt, 8 generated tokens (7 decode passes)"),
    "smol_b1": Workload("smol_b1", SMOL, batch=1, prompt_len=5, decode_steps=256),
    "smol_b16": Workload("smol_b16", SMOL.replace(max_batch=16, kv_dtype=DTYPE_BF16),
                         batch=16, prompt_len=512, decode_steps=512),
    "llama1b_b1": Workload("llama1b_b1", LLAMA1B.replace(max_batch=1), batch=1,
                           prompt_len=2048, decode_steps=256),
    "llama1b_b8": Workload("llama1b_b8", LLAMA1B, batch=8, prompt_len=2048,
                           decode_steps=256),
    "llama1b_long": Workload("llama1b_long", LLAMA1B.replace(max_batch=4, max_seq=32832),
                             batch=4, prompt_len=32768, decode_steps=64),
    # The long-context workload's attention at full size with a model small enough for
    # the oracle to prefill 4 x 32,768 positions offline: the Llama-3.2-1B attention
    # geometry (32 query heads, 8 kv heads, head_dim 64, dim 2048, theta 500000, bf16
    # KV) in 2 layers, with a small FFN and vocabulary.
    "llama1b_long_2l": Workload("llama1b_long_2l", LONG_2L, batch=4, prompt_len=32768,
                                decode_steps=8,
                                note="Llama-3.2-1B attention geometry, 2 layers, hidden 512, "
                                     "vocab 2048: 4 x 32768-token prompts + 8 decode steps"),
}


def layout(s: Shape) -> List[Tuple[str, int, int, int]]:
    """(name, layer, offset, count) of every tensor in canonical order, in elements.

    ``layer`` is -1 for the embedding and the output norm.
    """
    out = []
    off = 0

    def add(name, layer, count):
        nonlocal off
        out.append((name, layer, off, count))
        off += count

    qd = s.n_heads * s.head_dim
    kvd = s.n_kv_heads * s.head_dim
    add("token_emb", -1, s.vocab * s.dim)
    for l in range(s.n_layers):
        add("attn_norm", l, s.dim)
        add("wq", l, qd * s.dim)
        add("wk", l, kvd * s.dim)
        add("wv", l, kvd * s.dim)
        add("wo", l, s.dim * qd)
        add("ffn_norm", l, s.dim)
        add("w1", l, s.hidden * s.dim)
        add("w3", l, s.hidden * s.dim)
        add("w2", l, s.dim * s.hidden)
    add("output_norm", -1, s.dim)
    return out


def n_params(s: Shape) -> int:
    """Total number of stored weight elements (norm gains included)."""
    name, layer, off, count = layout(s)[-1]
    return off + count


def tensor(weights: np.ndarray, s: Shape, name: str, layer: int = -1) -> np.ndarray:
    """A view of one tensor of a canonical buffer (1-D, in storage dtype)."""
    for n, l, off, count in layout(s):
        if n == name and l == layer:
            return weights[off:off + count]
    raise KeyError((name, layer))


def f32_to_bf16_rne(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 bit patterns (uint16), nearest-even. Finite inputs only."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    u = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (u >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (the bits become the top half of the word)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


_ONE_BF16 = np.uint16(0x3F80)


def make_weights(s: Shape, seed: int = WEIGHT_SEED, std: float = 0.02) -> np.ndarray:
    """The canonical weight buffer: float32 array, or uint16 (bf16 bits) array."""
    total = n_params(s)
    bf16 = s.weight_dtype == DTYPE_BF16
    buf = np.empty(total, dtype=np.uint16 if bf16 else np.float32)
    rng = np.random.default_rng(seed)
    scale = np.float32(std)
    for name, _layer, off, count in layout(s):
        if name.endswith("norm"):
            buf[off:off + count] = _ONE_BF16 if bf16 else np.float32(1.0)
            continue
        # draw in chunks to bound the fp32 temporary
        done = 0
        while done < count:
            n = min(count - done, 1 << 26)
            vals = rng.standard_normal(n, dtype=np.float32) * scale
            buf[off + done:off + done + n] = f32_to_bf16_rne(vals) if bf16 else vals
            done += n
    return buf


def make_prompt(s: Shape, row: int, n: int, seed: int = PROMPT_SEED) -> np.ndarray:
    """Seeded uniform token ids in [0, vocab) for batch row ``row``."""
    return np.random.default_rng(seed + row).integers(0, s.vocab, n, dtype=np.int32)


def digest(a: np.ndarray) -> str:
    """sha256 of an array's bytes, used to check that two machines made the same input."""
    return hashlib.sha256(np.ascontiguousarray(a).view(np.uint8)).hexdigest()


def weight_bytes(s: Shape) -> int:
    return n_params(s) * (2 if s.weight_dtype == DTYPE_BF16 else 4)
