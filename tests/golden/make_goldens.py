"""Write the oracle's expected values for the large workloads.

The single-threaded fp32 oracle needs about 1 s per token position at the Llama-3.2-1B
shape (0.2 s at the SmolLM2 shape), so a 2048-token prompt plus 256 greedy decode steps
takes about half an hour per row: too slow to recompute inside a test.  This script runs
it once per row (rows in parallel, spawned processes) and stores, for the prefill's last
position and for every decode step:
the oracle's greedy id, its top-2 logit gap, max|logit|, its 8 largest logits with their
indices, and the logits at 64 fixed vocabulary indices; plus the whole logits vector at a
few positions (`full_steps`: the prefill, the first, a middle and the last decode step;
every step for the reduced long-context workload).  It calls only `oracle` and
`synth`.  The first 2048 tokens of the long-context workload's row 0 equal this row 0
prompt (the prompt generator draws sequentially), so the same file also pins that
workload's prefix.

Usage: python tests/golden/make_goldens.py WORKLOAD [rows...]
  llama1b_b8 0 1   -> llama1b_row0.npz, llama1b_row1.npz (also the llama1b_b1 row 0)
  smol_b16 0 7 15  -> smol_b16_row{0,7,15}.npz
  llama1b_long_2l 0 1 2 3 -> long2l_row{0..3}.npz (4 x 32768-token prefills, ~1 h per row)
"""
import multiprocessing as mp
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

PREFIX = {"llama1b_b8": "llama1b", "smol_b16": "smol_b16", "llama1b_long_2l": "long2l"}
SAMPLE_SEED = 4242
N_SAMPLE = 64
TOPK = 8


def sample_indices(vocab):
    return np.sort(np.random.default_rng(SAMPLE_SEED).choice(vocab, N_SAMPLE, replace=False)).astype(np.int32)


def full_steps(steps):
    """Record indices (0 = the prefill's last position) whose whole logits are stored."""
    if steps <= 16:
        return list(range(steps + 1))
    return [0, 1, steps // 2, steps]


def run_row(args):
    workload, row = args
    import oracle
    wl = synth.WORKLOADS[workload]
    s = wl.shape.replace(max_batch=1)
    W = synth.make_weights(s)
    prompt = synth.make_prompt(s, row, wl.prompt_len)
    idx = sample_indices(s.vocab)
    m = oracle.Model(s, W)
    out = {k: [] for k in ("ids", "gap", "maxabs", "top_idx", "top_val", "sampled", "full")}
    keep = set(full_steps(wl.decode_steps))

    def record(lg, nid):
        if len(out["ids"]) in keep:
            out["full"].append(lg.copy())
        top = np.argsort(-lg, kind="stable")[:TOPK]
        part = np.partition(lg, -2)[-2:]
        out["ids"].append(nid)
        out["gap"].append(float(part[1] - part[0]))
        out["maxabs"].append(float(np.abs(lg).max()))
        out["top_idx"].append(top.astype(np.int32))
        out["top_val"].append(lg[top])
        out["sampled"].append(lg[idx])

    t0 = time.time()
    lg, nid = m.prefill(0, prompt)
    record(lg, nid)
    print(f"row {row}: prefill {time.time() - t0:.0f}s", flush=True)
    for step in range(wl.decode_steps):
        lgs, ids = m.decode_step([0], [out["ids"][-1]], [wl.prompt_len + step])
        record(lgs[0], int(ids[0]))
        if step % 32 == 0 or wl.decode_steps <= 16:
            print(f"row {row}: step {step} {time.time() - t0:.0f}s", flush=True)
    m.close()
    res = {k: np.asarray(v) for k, v in out.items()}
    res["full_steps"] = np.asarray(full_steps(wl.decode_steps), dtype=np.int32)
    res["sample_idx"] = idx
    res["weights_sha256"] = np.array(synth.digest(W))
    res["prompt"] = prompt
    path = os.path.join(HERE, f"{PREFIX[workload]}_row{row}.npz")
    np.savez_compressed(path, **res)
    return path


if __name__ == "__main__":
    workload = sys.argv[1]
    rows = [int(r) for r in sys.argv[2:]] or [0]
    with mp.get_context("spawn").Pool(len(rows)) as pool:
        for p in pool.map(run_row, [(workload, r) for r in rows]):
            print("wrote", p)
