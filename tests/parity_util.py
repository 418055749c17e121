"""Shared helpers for the parity tests: oracle reference runs (optionally in parallel
processes) and the comparison rules.

Parity protocol: the oracle decodes greedily; its ids are fed to the GPU engine step by
step (teacher forcing), so both sides always see identical inputs.  Logits must agree
within ``tol * max|oracle logit|`` per (row, step): tol = 1e-3 with an fp32 KV cache,
2e-2 with a bf16 one.  A GPU id must equal the oracle id whenever the oracle's top-2
gap exceeds 1e-2 (GOTOken, "Building it one piece at a time": check the size of the
differences and whether they change the greedy token).
"""
from __future__ import annotations

import multiprocessing as mp
from typing import Dict, List, Sequence

import numpy as np

import synth

GAP = 1e-2


def tolerance(shape) -> float:
    return 2e-2 if shape.kv_dtype == synth.DTYPE_BF16 else 1e-3


def _oracle_job(args):
    shape, seed, prompts, steps, rows = args
    import oracle
    W = synth.make_weights(shape, seed=seed)
    ids, logs = oracle.greedy_run(shape, W, prompts, steps, rows=rows)
    return ids, logs


def oracle_reference(shape, prompts: Sequence[np.ndarray], steps: int, rows: List[int],
                     seed: int = synth.WEIGHT_SEED, procs: int = 1):
    """Greedy oracle runs of the given rows; returns (ids, logits) dicts keyed by row.

    Rows are independent sequences, so ``procs > 1`` splits them over spawned processes
    (each rebuilds the seeded weights itself).
    """
    if procs <= 1 or len(rows) == 1:
        return _oracle_job((shape.replace(max_batch=len(rows)), seed, prompts, steps, rows))
    ctx = mp.get_context("spawn")
    jobs = [(shape.replace(max_batch=1), seed, prompts, steps, [r]) for r in rows]
    ids: Dict[int, list] = {}
    logs: Dict[int, list] = {}
    with ctx.Pool(min(procs, len(jobs))) as pool:
        for i_, l_ in pool.map(_oracle_job, jobs):
            ids.update(i_)
            logs.update(l_)
    return ids, logs


def top2_gap(x: np.ndarray) -> float:
    part = np.partition(x, -2)[-2:]
    return float(part[1] - part[0])


def check_logits(gpu: np.ndarray, ref: np.ndarray, tol: float, what: str):
    scale = float(np.abs(ref).max())
    err = float(np.abs(gpu.astype(np.float64) - ref.astype(np.float64)).max())
    assert err <= tol * scale, f"{what}: max|d logit| = {err:.3e} > {tol} * {scale:.3e}"
    return err / scale


def check_id(gpu_id: int, ref_logits: np.ndarray, ref_id: int, what: str):
    if top2_gap(ref_logits) > GAP:
        assert gpu_id == ref_id, f"{what}: id {gpu_id} != oracle {ref_id} (gap {top2_gap(ref_logits):.3g})"
    else:
        # several ids are acceptable; the GPU one must be within the gap of the best
        assert ref_logits[gpu_id] >= ref_logits.max() - GAP, f"{what}: id {gpu_id} not near the top"


def gpu_teacher_forced(engine, shape, prompts, ref_ids: Dict[int, list], steps: int, rows_all: int,
                       collect_rows: Sequence[int]):
    """Prefill rows 0..rows_all-1, then ``steps`` batched decode steps.

    Rows in ``ref_ids`` are fed the oracle's ids; the others are fed their own GPU ids.
    Returns (logits, ids) dicts for ``collect_rows``: logits[r][s] is step s's vector
    (s = 0 is the prefill's last position).
    """
    import torch
    dev = torch.device("cuda")
    logits = {r: [] for r in collect_rows}
    ids = {r: [] for r in collect_rows}
    cur = {}
    for r in range(rows_all):
        lg, nid = engine.prefill_checked(r, prompts[r], want_logits=r in collect_rows)
        g = int(nid.item())
        if r in collect_rows:
            logits[r].append(lg.cpu().numpy())
            ids[r].append(g)
        cur[r] = ref_ids[r][0] if r in ref_ids else g
    seqs = list(range(rows_all))
    for s in range(steps):
        toks = torch.tensor([cur[r] for r in seqs], dtype=torch.int32, device=dev)
        poss = [len(prompts[r]) + s for r in seqs]
        lg, nid = engine.decode_checked(seqs, toks, poss, want_logits=True)
        nid = nid.cpu().numpy()
        lgn = None
        for i, r in enumerate(seqs):
            if r in collect_rows:
                if lgn is None:
                    lgn = lg.cpu().numpy()
                logits[r].append(lgn[i])
                ids[r].append(int(nid[i]))
            cur[r] = ref_ids[r][s + 1] if r in ref_ids else int(nid[i])
    rc = engine.sync()
    assert rc == 0, f"device status {rc}: {engine.last_error()}"
    return logits, ids


def compare_runs(shape, ref_ids, ref_logits, gpu_logits, gpu_ids, rows, label: str):
    tol = tolerance(shape)
    worst = 0.0
    for r in rows:
        assert len(gpu_logits[r]) == len(ref_logits[r])
        for s, (g, o) in enumerate(zip(gpu_logits[r], ref_logits[r])):
            worst = max(worst, check_logits(g, o, tol, f"{label} row {r} step {s}"))
            check_id(gpu_ids[r][s], o, ref_ids[r][s], f"{label} row {r} step {s}")
    return worst
