"""Reference sampling of the next token from one row of logits (fp64, plain loops).

TEST INFRASTRUCTURE ONLY: imported by ``tests/`` (never by the CUDA library or its
binding).

The procedure is the one on "Inside nanochat Part 4: Understanding Inference" (The
Sampling Function, Greedy Decoding, Temperature Sampling, Top-K Filtering):

* temperature 0: greedy, the index of the largest logit (the lowest index on ties);
* top-k (k >= 1): keep the k largest logits (sorted largest first, ties by lower
  index), divide them by the temperature, softmax over them, draw one;
* no top-k (k = 0): divide every logit by the temperature, softmax over the whole
  vocabulary in index order, draw one.

Top-p appears on the kasahare 0.4.0 page only as a CLI flag beside top-k ("CLI flags",
--top-p 0.95 with --top-k 40); it is read here as nucleus filtering applied after top-k:
keep the shortest prefix of the sorted candidates whose probability reaches p, and
renormalise over it.  It needs k >= 1.

The draw: the page draws with torch.multinomial and a seeded generator.  Here the
uniform variate u in [0, 1) is an input (one per row), and the draw is the inverse of
the cumulative distribution over the candidates in the order above: the first
candidate whose running sum of weights exceeds u times the total.
"""
from __future__ import annotations

import math
from typing import List, Tuple

import numpy as np


def candidates(logits, temperature: float, top_k: int, top_p: float) -> Tuple[List[int], List[float]]:
    """The candidate ids in draw order and their unnormalised weights (fp64)."""
    x = [float(v) for v in np.asarray(logits, dtype=np.float32)]
    V = len(x)
    if top_k >= 1:
        k = min(top_k, V)
        order = sorted(range(V), key=lambda i: (-x[i], i))[:k]
    else:
        if top_p < 1.0:
            raise ValueError("top-p needs top-k >= 1")
        order = list(range(V))
    vals = [x[i] / temperature for i in order]
    m = max(vals)
    w = [math.exp(v - m) for v in vals]
    if top_p < 1.0:
        total = math.fsum(w)
        run, keep = 0.0, len(w)
        for i, wi in enumerate(w):
            run += wi
            if run >= top_p * total:
                keep = i + 1
                break
        order, w = order[:keep], w[:keep]
    return order, w


def sample(logits, temperature: float, top_k: int, top_p: float, u: float) -> int:
    """The sampled token id of one row."""
    x = np.asarray(logits, dtype=np.float32)
    if temperature == 0.0:
        best = 0
        for i in range(1, len(x)):
            if x[i] > x[best]:
                best = i
        return best
    order, w = candidates(x, temperature, top_k, top_p)
    total = 0.0
    for wi in w:
        total += wi
    target = u * total
    run = 0.0
    for i, wi in zip(order, w):
        run += wi
        if run > target:
            return i
    return order[-1]
