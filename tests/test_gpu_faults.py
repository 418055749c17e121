"""The failure paths, exercised without faulting the GPU.

* A hand-off that never arrives: slm_debug_faults shortens the device-side wait limit
  to tens of microseconds and makes one CTA skip one publish of the first layer's
  residual.  The consumers' bounded waits run out, the step finishes (no hang), a
  synchronous call reports SLM_ETIMEOUT itself, slm_sync reports and clears it, and the
  same context then decodes correctly again (checked against the oracle).  Both decode
  kernels: the cluster kernel (single-row steps) and the persistent one.
* An allocation that fails inside slm_create (SLM_FAULT_ALLOC_AFTER=n, read by the
  library at each device allocation): SLM_ENOMEM, nothing leaked, the next create works.
"""
import os

import numpy as np
import pytest

import synth
from parity_util import check_id, check_logits, oracle_reference, tolerance

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

SLM_ENOMEM, SLM_ETIMEOUT = -2, -7


@pytest.fixture(scope="module")
def slm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import llama_decode_kv_gb300 as m
    return m


SHAPE = synth.TINY.replace(max_batch=2, max_seq=48, weight_dtype=synth.DTYPE_BF16)


def _engine(slm, cluster: bool):
    W = synth.make_weights(SHAPE, seed=21)
    old = os.environ.get("SLM_NO_CLUSTER")
    try:
        if not cluster:
            os.environ["SLM_NO_CLUSTER"] = "1"
        eng = slm.Engine(SHAPE, W)
    finally:
        if old is None:
            os.environ.pop("SLM_NO_CLUSTER", None)
        else:
            os.environ["SLM_NO_CLUSTER"] = old
    assert (eng.cluster_plan() is not None) == cluster
    return eng


@pytest.mark.parametrize("kernel", ["cluster", "persistent"])
def test_lost_publish_times_out_and_recovers(slm, kernel):
    eng = _engine(slm, kernel == "cluster")
    dev = torch.device("cuda")
    prompt = synth.make_prompt(SHAPE, 0, 6)
    steps = 4
    ref_ids, ref_logits = oracle_reference(SHAPE, [prompt], steps, [0], seed=21)
    _, nid = eng.prefill_checked(0, prompt, want_logits=False)
    eng.debug_faults(wait_ns=50_000, lost_publish=1)
    # device buffers: the call returns at once, slm_sync sees the timeout
    tok = torch.tensor([ref_ids[0][0]], dtype=torch.int32, device=dev)
    ids = torch.empty(1, dtype=torch.int32, device=dev)
    assert eng.decode_step([0], tok, [6], None, ids) == 0
    assert eng.sync() == SLM_ETIMEOUT
    assert "timed out" in eng.last_error()
    assert eng.sync() == 0  # cleared
    # host buffers: the call waits for the step and reports the timeout itself
    host_ids = np.zeros(1, dtype=np.int32)
    rc = eng.decode_step([0], np.array([ref_ids[0][1]], dtype=np.int32), [7], None, host_ids)
    assert rc == SLM_ETIMEOUT, rc
    assert eng.sync() == SLM_ETIMEOUT
    # back to normal: the same context decodes this sequence again, against the oracle
    eng.debug_faults(wait_ns=0, lost_publish=0)
    eng.reset(0)
    lg, nid = eng.prefill_checked(0, prompt, want_logits=True)
    tol = tolerance(SHAPE)
    check_logits(lg.cpu().numpy(), ref_logits[0][0], tol, f"{kernel} prefill after the fault")
    check_id(int(nid.item()), ref_logits[0][0], ref_ids[0][0], f"{kernel} prefill after the fault")
    for st in range(steps):
        tok = torch.tensor([ref_ids[0][st]], dtype=torch.int32, device=dev)
        lg, ids = eng.decode_checked([0], tok, [6 + st], want_logits=True)
        check_logits(lg[0].cpu().numpy(), ref_logits[0][st + 1], tol, f"{kernel} step {st} after the fault")
        check_id(int(ids[0].item()), ref_logits[0][st + 1], ref_ids[0][st + 1], f"{kernel} step {st} after the fault")
    assert eng.sync() == 0, eng.last_error()
    eng.close()


def test_allocation_failure_in_create(slm):
    W = synth.make_weights(SHAPE, seed=21)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    os.environ["SLM_FAULT_ALLOC_AFTER"] = "3"
    try:
        with pytest.raises(slm.SlmError) as e:
            slm.Engine(SHAPE, W)
        assert e.value.code == SLM_ENOMEM
        assert "injected allocation failure" in str(e.value)
    finally:
        os.environ.pop("SLM_FAULT_ALLOC_AFTER", None)
    torch.cuda.synchronize()
    # what the failed create took was freed (allow the driver's own small variations)
    assert torch.cuda.mem_get_info()[0] >= free0 - (64 << 20)
    eng = slm.Engine(SHAPE, W)
    _, nid = eng.prefill_checked(0, synth.make_prompt(SHAPE, 0, 3), want_logits=False)
    assert eng.sync() == 0
    eng.close()
