#!/usr/bin/env python
"""Decode benchmark: greedy KV-cached decode on the SmolLM2-135M shape at batch 1 (headline),
with the other workloads in objects of the same line: SmolLM2 at batch 16 (`batch16`),
Llama-3.2-1B at batch 1 and 8 after 2048-token prompts and at batch 4 after 32768-token
prompts (`llama1b_b1`, `llama1b_b8`, `llama1b_long`).

``python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]``

One step = one ``slm_decode_step`` (every phase of the decode step for the batch) on
synthetic random-init bf16 weights (~N(0, 0.02)) and a seeded random 5-token prompt;
the next ids stay on the device and feed the following step.  Weights (269 MB) stream
from HBM every step and exceed the 129 MB L2, so no flush is needed between steps.
Prints one JSON line.  Under torchrun each rank runs an independent replica (the path
has no exchange step), the timed region is bracketed by barriers and the slowest
rank's time counts.  ``--impl reference`` times the CPU oracle on the host instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "decode tokens/sec at batch 1 and 16; achieved HBM GB/s vs ~8 TB/s peak"
UNIT = "tokens/s"
WORKLOAD = "smol_b1"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
KERNEL_SRC = os.path.join(ROOT, "llama_decode_kv_gb300", "csrc", "decode_cluster.cu")
PROFILE = os.path.join(ROOT, "profiles", "decode_cluster_kernel.smol_b1.txt")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def peaks_tensor():
    """bf16 tensor peak for a kernel timed inside a long run of launches: the sustained
    figure (the burst one, or the fallback, when it is missing)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        if "bf16_tflops_sustained" in d:
            return float(d["bf16_tflops_sustained"]), "measured sustained"
        return float(d["bf16_tflops"]), "measured burst"
    except Exception:
        return 1700.0, "fallback sustained"


def host_cpu():
    """CPU model of this host and its logical core count."""
    model = None
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model")):
                model = line.split(":", 1)[1].strip()
                break
        if model is None:
            r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
            for line in r.stdout.splitlines():
                if line.startswith("Model name:"):
                    model = line.split(":", 1)[1].strip()
                    break
    except Exception:
        pass
    return {"cpu_model": model or "unknown", "nproc": os.cpu_count()}


class pinned_to_core0:
    """Run the enclosed (single-threaded) oracle pinned to core 0, like taskset -c 0."""

    def __enter__(self):
        try:
            self.old = os.sched_getaffinity(0)
            os.sched_setaffinity(0, {0})
            self.ok = True
        except Exception:
            self.ok = False
        return self

    def __exit__(self, *a):
        if self.ok:
            os.sched_setaffinity(0, self.old)


def kv_bytes_read(shape, ctx: int) -> int:
    """K and V bytes one row reads in one step at context length ctx (all layers)."""
    esz = 2 if shape.kv_dtype == synth.DTYPE_BF16 else 4
    return 2 * ctx * shape.head_dim * shape.n_kv_heads * esz * shape.n_layers


def profile_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it matches the source."""
    try:
        src = hashlib.sha256(open(KERNEL_SRC, "rb").read()).hexdigest()
        fields = {}
        for line in open(PROFILE):
            if ":" in line:
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
        if fields.get("kernel_source_sha256") != src:
            return None
        return float(fields["dram_bytes_per_launch"])
    except Exception:
        return None


class Clocks:
    """nvidia-smi samples during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo")
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def prefill_measure(slm, torch, W, local: int, reps: int = 3):
    """Tensor-core prefill of a 512-token prompt on the same weights with a bf16 KV cache
    (the SmolLM2 batch-16 workload's prompt length); FLOPs counted once per MAC of the
    linear layers and the logits row plus causal attention."""
    s = synth.WORKLOADS["smol_b16"].shape.replace(max_batch=1)
    eng = slm.Engine(s, W)
    n = 512
    prompt = torch.as_tensor(synth.make_prompt(s, 0, n)).to(torch.device("cuda", local))
    nid = torch.empty(1, dtype=torch.int32, device=prompt.device)
    times = []
    for i in range(reps + 1):
        eng.reset(0)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        rc = eng.prefill(0, prompt, None, nid)
        b.record()
        torch.cuda.synchronize()
        if rc != 0:
            raise RuntimeError(f"slm_prefill: {eng.last_error()}")
        if i:
            times.append(a.elapsed_time(b) / 1e3)
    assert eng.sync() == 0, eng.last_error()
    eng.close()
    t = statistics.median(times)
    lin = synth.n_params(s) - s.vocab * s.dim  # matrices of the blocks
    flops = 2.0 * lin * n + 2.0 * s.vocab * s.dim + 2.0 * 2 * s.head_dim * s.n_heads * s.n_layers * n * (n + 1) / 2
    return t, flops


def paged_measure(slm, torch, W, local: int, steps: int, warmup: int, page: int = 64):
    """The headline workload on a paged KV cache (`page`-position pages): the same prompt,
    warm-up and number of steps as the main timed region, so the same contexts; device
    ids fed back.  Returns ms per step (the overhead of the page table is the ratio to
    the contiguous cache's)."""
    wl = synth.WORKLOADS[WORKLOAD]
    s = wl.shape
    dev = torch.device("cuda", local)
    eng = slm.Engine(s, W, kv_page_size=page)
    toks = [torch.zeros(1, dtype=torch.int32, device=dev) for _ in range(2)]
    prompt = synth.make_prompt(s, 0, wl.prompt_len)
    _, nid = eng.prefill_checked(0, prompt, want_logits=False)
    toks[0].copy_(nid)
    pos, cur = len(prompt), 0
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(warmup + steps):
        if i == warmup:
            torch.cuda.synchronize()
            a.record(stream)
        if eng.decode_step([0], toks[cur], [pos], None, toks[1 - cur]) != 0:
            raise RuntimeError(f"paged decode: {eng.last_error()}")
        pos, cur = pos + 1, 1 - cur
    b.record(stream)
    torch.cuda.synchronize()
    if eng.sync() != 0:
        raise RuntimeError(f"device status after the paged run: {eng.last_error()}")
    eng.close()
    return a.elapsed_time(b) / steps


def batch16_measure(slm, torch, W, local: int, warmup: int = 3):
    """The SmolLM2 batch-16 workload: 16 independent rows with a bf16 KV cache, each
    prefilled with a seeded 512-token prompt (tensor-core prefill, untimed), then batched
    greedy decode steps up to context 1024, timed with CUDA events on the launching
    stream.  HBM bytes per step = the weights once + every row's K and V reads."""
    wl = synth.WORKLOADS["smol_b16"]
    s, B = wl.shape, wl.batch
    eng = slm.Engine(s, W)  # the weights do not depend on the batch or the cache type
    dev = torch.device("cuda", local)
    toks = [torch.empty(B, dtype=torch.int32, device=dev) for _ in range(2)]
    rows = list(range(B))
    # the 16 prompts prefilled in one call (GEMMs over all 8,192 positions), timed
    prompts = torch.as_tensor(np.concatenate([synth.make_prompt(s, r, wl.prompt_len) for r in rows])).to(dev)
    pa, pb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pf_ms = []
    for rep in range(3):
        eng.reset(-1)
        torch.cuda.synchronize()
        pa.record(torch.cuda.current_stream())
        rc = eng.prefill_batch(rows, prompts, [wl.prompt_len] * B, None, toks[0])
        pb.record(torch.cuda.current_stream())
        torch.cuda.synchronize()
        if rc != 0:
            raise RuntimeError(f"slm_prefill_batch: {eng.last_error()}")
        pf_ms.append(pa.elapsed_time(pb))
    state = {"pos": wl.prompt_len, "cur": 0, "ctx": []}

    def step():
        c = state["cur"]
        rc = eng.decode_step(rows, toks[c], [state["pos"]] * B, None, toks[1 - c])
        if rc != 0:
            raise RuntimeError(f"slm_decode_step: {eng.last_error()}")
        state["ctx"].append(state["pos"] + 1)
        state["pos"] += 1
        state["cur"] = 1 - c

    for _ in range(warmup):
        step()
    state["ctx"].clear()
    n = s.max_seq - state["pos"]
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(n):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    if eng.sync() != 0:
        raise RuntimeError(f"device status after the batch-16 run: {eng.last_error()}")
    eng.close()
    bytes_step = sum(synth.weight_bytes(s) + B * kv_bytes_read(s, c) for c in state["ctx"]) / n
    # on-device sampling of the same batch: temperature 0.8, top-k 40, top-p 0.95 over
    # seeded logits of the vocabulary's size, one uniform per row
    g = torch.Generator(device=dev).manual_seed(1234)
    lg = torch.randn((B, s.vocab), generator=g, device=dev) * 2.0
    us = torch.rand((B,), generator=g, device=dev)
    ids = torch.empty(B, dtype=torch.int32, device=dev)
    for _ in range(3):
        slm.sample(lg, 0.8, 40, 0.95, us, ids)
    reps = 50
    a.record(stream)
    for _ in range(reps):
        rc = slm.sample(lg, 0.8, 40, 0.95, us, ids)
    b.record(stream)
    torch.cuda.synchronize()
    if rc != 0:
        raise RuntimeError("slm_sample failed")
    samp_us = a.elapsed_time(b) / reps * 1e3
    return {"workload": "smol_b16: SmolLM2-135M shape, bf16 KV cache, 16 rows x 512-token prompt, greedy decode "
                        f"to context {s.max_seq}",
            "tokens_per_s": B * n / (ms / 1e3), "ms_per_step": ms / n, "steps": n, "warmup": warmup,
            "contexts": [min(state["ctx"]), max(state["ctx"])], "bytes_per_step": bytes_step,
            "hbm_gbs": bytes_step / (ms / 1e3 / n) / 1e9,
            "prefill": {"call": "slm_prefill_batch, 16 prompts x 512 tokens", "ms": min(pf_ms[1:]),
                        "tokens_per_s": B * wl.prompt_len / (min(pf_ms[1:]) / 1e3)},
            "sampling": {"call": "slm_sample, 16 rows x 49152 logits, temperature 0.8, top-k 40, top-p 0.95",
                         "us_per_call": samp_us,
                         "logit_gbs": B * s.vocab * 4 / (samp_us / 1e6) / 1e9}}


def cpu_baseline(shape, W, prompt, budget_s: float):
    """The oracle, as it stands, on the host (pinned to core 0): greedy decode steps
    after the prompt, the prefill timed per token."""
    import oracle
    with pinned_to_core0() as pin:
        m = oracle.Model(shape, W)
        t0 = time.perf_counter()
        _, nid = m.prefill(0, prompt)
        pf_s = time.perf_counter() - t0
        steps, pos = 0, len(prompt)
        t0 = time.perf_counter()
        while True:
            _, ids = m.decode_step([0], [nid], [pos])
            nid, pos, steps = int(ids[0]), pos + 1, steps + 1
            if time.perf_counter() - t0 >= budget_s or pos >= shape.max_seq:
                break
        dt = time.perf_counter() - t0
        m.close()
    return {"value": steps / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "pinned": "core 0" if pin.ok else "not pinned", **host_cpu(),
            "ms_per_step": dt / steps * 1e3, "ms_per_prefill_token": pf_s / len(prompt) * 1e3,
            "sample": f"{steps} single-threaded oracle decode steps (contexts {len(prompt) + 1}.."
                      f"{pos}) after a {len(prompt)}-token prompt, SmolLM2-135M shape, batch 1"}


def oracle_llama_sample(shape, W, n_prompt: int = 3, n_steps: int = 2):
    """The oracle on the Llama-3.2-1B shape, pinned to core 0: a short prompt and a few
    decode steps (labelled sampled: the 2048- and 32768-token prefills are far beyond a
    benchmark's time on one core; per step the weights dominate, about 1.24 GMAC)."""
    import oracle
    s = shape.replace(max_batch=1, max_seq=16)
    with pinned_to_core0() as pin:
        m = oracle.Model(s, W)
        prompt = synth.make_prompt(s, 0, n_prompt)
        t0 = time.perf_counter()
        _, nid = m.prefill(0, prompt)
        pf_s = time.perf_counter() - t0
        pos = n_prompt
        t0 = time.perf_counter()
        for _ in range(n_steps):
            _, ids = m.decode_step([0], [nid], [pos])
            nid, pos = int(ids[0]), pos + 1
        dt = time.perf_counter() - t0
        m.close()
    return {"kind": "oracle", "cores": 1, "pinned": "core 0" if pin.ok else "not pinned",
            "ms_per_step_per_row": dt / n_steps * 1e3, "ms_per_prefill_token": pf_s / n_prompt * 1e3,
            "sample": f"sampled: {n_steps} decode steps at contexts {n_prompt + 1}..{pos} after a "
                      f"{n_prompt}-token prompt (not at the workload's context)"}


def llama_measure(slm, torch, W, local: int, name: str, steps: int, warmup: int = 3, peak: float = 0.0):
    """A Llama-3.2-1B workload (bf16 weights and KV cache): every row prefilled with its
    seeded prompt in one batched tensor-core prefill (timed separately), then `steps`
    batched greedy decode steps timed with CUDA events.  HBM bytes per step = the
    weights once + every row's K and V reads at that step's context."""
    wl = synth.WORKLOADS[name]
    s, B = wl.shape, wl.batch
    dev = torch.device("cuda", local)
    eng = slm.Engine(s, W)
    rows = list(range(B))
    prompts = torch.as_tensor(np.concatenate([synth.make_prompt(s, r, wl.prompt_len) for r in rows])).to(dev)
    toks = [torch.empty(B, dtype=torch.int32, device=dev) for _ in range(2)]
    pa, pb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    pa.record(torch.cuda.current_stream())
    rc = eng.prefill_batch(rows, prompts, [wl.prompt_len] * B, None, toks[0])
    pb.record(torch.cuda.current_stream())
    torch.cuda.synchronize()
    if rc != 0:
        raise RuntimeError(f"{name} prefill: {eng.last_error()}")
    pf_ms = pa.elapsed_time(pb)
    state = {"pos": wl.prompt_len, "cur": 0, "ctx": []}

    def step():
        c = state["cur"]
        if eng.decode_step(rows, toks[c], [state["pos"]] * B, None, toks[1 - c]) != 0:
            raise RuntimeError(f"{name} decode: {eng.last_error()}")
        state["ctx"].append(state["pos"] + 1)
        state["pos"] += 1
        state["cur"] = 1 - c

    for _ in range(warmup):
        step()
    state["ctx"].clear()
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    if eng.sync() != 0:
        raise RuntimeError(f"device status after {name}: {eng.last_error()}")
    eng.close()
    bytes_step = sum(synth.weight_bytes(s) + B * kv_bytes_read(s, c) for c in state["ctx"]) / steps
    gbs = bytes_step / (ms / 1e3 / steps) / 1e9
    pf_tokens = B * wl.prompt_len
    return {"workload": f"{name}: Llama-3.2-1B shape (dim 2048, 16 layers, 32/8 heads, hidden 8192, vocab "
                        f"128256), bf16 weights and KV cache, {B} x {wl.prompt_len}-token prompt, greedy decode",
            "tokens_per_s": B * steps / (ms / 1e3), "ms_per_step": ms / steps, "steps": steps, "warmup": warmup,
            "contexts": [min(state["ctx"]), max(state["ctx"])], "bytes_per_step": bytes_step,
            "hbm_gbs": gbs, "roofline_frac": gbs / peak if peak else None, "peak_gbs": peak,
            "prefill": {"call": f"slm_prefill_batch, {B} x {wl.prompt_len} tokens", "ms": pf_ms,
                        "tokens_per_s": pf_tokens / (pf_ms / 1e3)}}


def q8_weight_bytes(s) -> int:
    """Device bytes of block-quantised int8 weights: every matrix row stores one byte per
    weight plus a 4-byte scale per block of 32; the norm gains stay fp32."""
    total = 0
    for name, _layer, _off, count in synth.layout(s):
        if name.endswith("norm"):
            total += 4 * count
            continue
        k = s.hidden if name == "w2" else (s.n_heads * s.head_dim if name == "wo" else s.dim)
        total += (count // k) * (k + 4 * ((k + 31) // 32))
    return total


def q8_measure(slm, torch, local: int, base, prompt_len: int, steps: int, peak: float, warmup: int = 3):
    """Batch-1 greedy decode with block-quantised int8 weights (slm_config.weight_dtype =
    SLM_Q8): the prompt is prefilled one position at a time (untimed), then `steps` steps
    timed with CUDA events, ids fed back on the device.  Bytes per step = the int8 weights
    and scales once + the K and V rows read."""
    s = base.replace(weight_dtype=synth.DTYPE_Q8, max_batch=1)
    W = synth.make_weights(s)  # fp32, quantised by slm_create
    dev = torch.device("cuda", local)
    eng = slm.Engine(s, W)
    del W
    toks = [torch.zeros(1, dtype=torch.int32, device=dev) for _ in range(2)]
    _, nid = eng.prefill_checked(0, synth.make_prompt(s, 0, prompt_len), want_logits=False)
    toks[0].copy_(nid)
    pos, cur, ctx = prompt_len, 0, []
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(warmup + steps):
        if i == warmup:
            torch.cuda.synchronize()
            a.record(stream)
        if eng.decode_step([0], toks[cur], [pos], None, toks[1 - cur]) != 0:
            raise RuntimeError(f"int8 decode: {eng.last_error()}")
        if i >= warmup:
            ctx.append(pos + 1)
        pos, cur = pos + 1, 1 - cur
    b.record(stream)
    torch.cuda.synchronize()
    if eng.sync() != 0:
        raise RuntimeError(f"device status after the int8 run: {eng.last_error()}")
    eng.close()
    ms = a.elapsed_time(b) / steps
    bytes_step = q8_weight_bytes(s) + sum(kv_bytes_read(s, c) for c in ctx) / steps
    gbs = bytes_step / (ms / 1e3) / 1e9
    return {"ms_per_step": ms, "tokens_per_s": 1e3 / ms, "steps": steps, "contexts": [min(ctx), max(ctx)],
            "bytes_per_step": bytes_step, "hbm_gbs": gbs, "roofline_frac": gbs / peak, "peak_gbs": peak}


def run_reference(args, world, rank):
    if rank != 0:
        return
    wl = synth.WORKLOADS[WORKLOAD]
    s = wl.shape
    W = synth.make_weights(s)
    prompt = synth.make_prompt(s, 0, wl.prompt_len)
    import oracle
    m = oracle.Model(s, W)
    _, nid = m.prefill(0, prompt)
    pos = len(prompt)
    for _ in range(args.warmup):
        _, ids = m.decode_step([0], [nid], [pos])
        nid, pos = int(ids[0]), pos + 1
    t0 = time.perf_counter()
    steps = 0
    cap_s = 150.0
    while steps < args.steps and pos < s.max_seq:
        _, ids = m.decode_step([0], [nid], [pos])
        nid, pos, steps = int(ids[0]), pos + 1, steps + 1
        if time.perf_counter() - t0 > cap_s:
            break
    dt = time.perf_counter() - t0
    value = steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": steps, "warmup": args.warmup, "ms_per_step": dt / steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: SmolLM2-135M shape, batch 1, 5-token prompt, greedy "
                               "decode", "batch": 1, "weights": "bf16", "kv": "f32"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{steps} oracle decode steps after {args.warmup} warm-up steps"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    import torch

    import llama_decode_kv_gb300 as slm

    torch.cuda.set_device(local)
    wl = synth.WORKLOADS[WORKLOAD]
    s = wl.shape
    W = synth.make_weights(s)
    prompt = synth.make_prompt(s, rank, wl.prompt_len)
    eng = slm.Engine(s, W)
    dev = torch.device("cuda", local)
    toks = [torch.zeros(1, dtype=torch.int32, device=dev) for _ in range(2)]
    _, nid = eng.prefill_checked(0, prompt, want_logits=False)
    toks[0].copy_(nid)
    state = {"pos": len(prompt), "cur": 0, "ctx": []}

    def step():
        if state["pos"] >= s.max_seq:  # wrap: the sequence starts over (host-side reset)
            eng.reset(0)
            state["pos"] = 0
        c = state["cur"]
        rc = eng.decode_step([0], toks[c], [state["pos"]], None, toks[1 - c])
        if rc != 0:
            raise RuntimeError(f"slm_decode_step: {slm.STATUS.get(rc)} {eng.last_error()}")
        state["ctx"].append(state["pos"] + 1)
        state["pos"] += 1
        state["cur"] = 1 - c

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    state["ctx"].clear()
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    clocks = Clocks(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    ev[0].record(stream)
    for i in range(args.steps):
        step()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(world)
    total_ms = ev[0].elapsed_time(ev[-1])
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    rc = eng.sync()
    if rc != 0:
        raise RuntimeError(f"device status after the timed region: {eng.last_error()}")
    t_max = max_over_ranks(total_ms, world)
    tokens = args.steps * wl.batch * world
    value = tokens / (t_max / 1e3)

    wbytes = synth.weight_bytes(s)
    alg_bytes = sum(wbytes + kv_bytes_read(s, c) for c in state["ctx"])
    per_launch_bytes = alg_bytes / args.steps
    per_launch_s = total_ms / 1e3 / args.steps
    achieved = per_launch_bytes / per_launch_s / 1e9
    peak, peak_kind = peaks()
    traffic = profile_traffic()

    # end to end through the C ABI with host buffers (copies inside the timed region), over
    # the same contexts as the device-timed steps: the sequence is prefilled again and
    # given the same warm-up
    eng.reset(0)
    _, nid = eng.prefill_checked(0, prompt, want_logits=False)
    tok_h = np.array([int(nid.item())], dtype=np.int32)
    ids_h = np.empty(1, dtype=np.int32)
    state["pos"] = len(prompt)
    for _ in range(max(args.warmup, 3)):
        if eng.decode_step([0], tok_h, [state["pos"]], None, ids_h) != 0:
            raise RuntimeError(f"slm_decode_step (host buffers): {eng.last_error()}")
        tok_h[0] = ids_h[0]
        state["pos"] += 1
    e2e_steps = args.steps
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        if state["pos"] >= s.max_seq:
            eng.reset(0)
            state["pos"] = 0
        rc = eng.decode_step([0], tok_h, [state["pos"]], None, ids_h)
        if rc != 0:
            raise RuntimeError(f"slm_decode_step (host buffers): {eng.last_error()}")
        tok_h[0] = ids_h[0]
        state["pos"] += 1
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e_value = e2e_steps * wl.batch * world / e2e_s

    eng.reset(0)
    paged_ms = paged_measure(slm, torch, W, local, args.steps, max(args.warmup, 3))
    pf_t, pf_flops = prefill_measure(slm, torch, W, local)
    tflops_peak, tflops_kind = peaks_tensor()
    b16 = batch16_measure(slm, torch, W, local)
    b16["roofline_frac"] = b16["hbm_gbs"] / peak
    b16["peak_gbs"] = peak
    cluster = eng.cluster_plan()
    eng.close()
    del W
    W_llama = synth.make_weights(synth.LLAMA1B)
    llama = {n: llama_measure(slm, torch, W_llama, local, n, st, peak=peak)
             for n, st in (("llama1b_b1", 64), ("llama1b_b8", 64), ("llama1b_long", 32))}
    q8 = {"what": "block-quantised int8 weights (SLM_Q8: blocks of 32 per row, fp32 scales), batch 1, "
                  "fp32 activations and accumulation, persistent kernel",
          "smol_b1_q8": q8_measure(slm, torch, local, synth.SMOL, wl.prompt_len, args.steps, peak),
          "llama1b_b1_q8": q8_measure(slm, torch, local, synth.LLAMA1B, 128, 64, peak)}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": t_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (random-init bf16 weights ~N(0,0.02), seeded random prompt)",
        "config": {
            "workload": f"{WORKLOAD}: SmolLM2-135M shape (dim 576, 30 layers, 9/3 heads, "
                        "hidden 1536, vocab 49152), batch 1, 5-token prompt, greedy decode",
            "batch": wl.batch, "weights": "bf16", "kv": "f32", "accumulate": "f32",
            "contexts": [min(state["ctx"]), max(state["ctx"])] if state["ctx"] else None,
            "l2": "inputs larger than L2: 269 MB of weights stream from HBM every step",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "latency_us": {"median": statistics.median(per) * 1e3,
                       "p10": float(np.percentile(per, 10)) * 1e3,
                       "p90": float(np.percentile(per, 90)) * 1e3},
        "bytes_per_step": per_launch_bytes,
        "hbm_gbs": achieved,
        "frac_of_8tbs": achieved / NOMINAL_HBM_GBS,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "decode_cluster_kernel" if cluster else "decode_step_kernel",
                     "peak_kind": peak_kind},
        "kernel_plan": cluster,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": 4 * wl.batch,
                "d2h_bytes_per_step": 4 * wl.batch},
        "gpu_launches": args.steps,
        "prefill": {"workload": "512-token prompt, same SmolLM2-135M-shaped weights, bf16 KV cache",
                    "tokens_per_s": 512 / pf_t, "ms": pf_t * 1e3,
                    "tflops": pf_flops / pf_t / 1e12, "peak_tflops": tflops_peak, "peak_kind": tflops_kind,
                    "frac": pf_flops / pf_t / 1e12 / tflops_peak, "bound": "tensor",
                    "note": "activation operands split into bf16 hi + lo: the tensor cores execute 2x these FLOPs"},
        "paged": {"what": "the same workload, steps and contexts on a paged KV cache (64-position pages, "
                          "slm_config.kv_page_size = 64)",
                  "ms_per_step": paged_ms, "tokens_per_s": wl.batch * 1e3 / paged_ms,
                  "overhead_vs_contiguous": paged_ms / (total_ms / args.steps) - 1.0},
        "batch16": b16,
        "int8_weights": q8,
        **llama,
        "clocks": clk,
    }
    if world == 1:
        line["cpu_baseline"] = cpu_baseline(s, synth.make_weights(s), prompt, args.cpu_budget)
        lo = oracle_llama_sample(synth.LLAMA1B, W_llama)
        for n in llama:
            line[n]["cpu_baseline"] = lo
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world, rank, local = dist_init()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
