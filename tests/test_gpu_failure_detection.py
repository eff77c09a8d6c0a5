"""Failure detection without a GPU fault.

* A bounded wait that runs out: the test hook kda_set_test_fault(KDA_TEST_FAULT_STALL_RECORD_INPUTS) makes
  the prep kernel issue no input copies, so its first wait finds nothing to wait for; it gives up after a
  short poll, flags KDA_DEV_TIMEOUT and returns with nothing in flight.  The call completes, nothing is
  written, and the context stays usable (a normal prefill right after matches the oracle).
* The debug mode of the C ABI (kda_set_debug_checks): calls that break the slot-id contract (a repeated
  slot id, a copy whose destination is its own source, a snapshot into a slot the prefill also owns) are
  rejected on the host with KDA_ERR_INVALID_ARG before anything is enqueued, so the pool is untouched."""
import numpy as np
import pytest
import torch

import synth
from tests._gpu import PrefillRun, dev, oracle_prefill, host, rel_err, status

pytestmark = pytest.mark.gpu

INVALID_ARG = 1


@pytest.fixture
def debug(cuda):
    was = cuda.kda_debug_checks()
    cuda.kda_set_debug_checks(True)
    yield cuda
    cuda.kda_set_debug_checks(was)


def test_debug_mode_rejects_repeated_decode_slots(debug):
    kda = debug
    p = synth.decode_verify(B=6, W=2, H=2, d=32, num_slots=10, dtype=synth.F32)
    q, k, v, g, beta = dev(p.q), dev(p.k), dev(p.v), dev(p.g), dev(p.beta)
    pool = dev(p.pool)
    pool0 = pool.clone()
    out = torch.zeros(p.B, p.H, p.dv, device="cuda")
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    ids = p.slot_ids.copy()
    ids[4] = ids[1]
    with pytest.raises(kda.KdaError) as e:
        kda.kda_decode_step(q, k, v, g, beta, pool, dev(ids), out, dev_status=st)
    assert e.value.code == INVALID_ARG
    torch.cuda.synchronize()
    assert torch.equal(pool, pool0) and status(st) == (0, 0)
    kda.kda_decode_step(q, k, v, g, beta, pool, dev(p.slot_ids), out, dev_status=st)  # distinct: accepted
    torch.cuda.synchronize()
    assert status(st) == (0, p.B * p.H)


def test_debug_mode_rejects_aliased_copies(debug):
    kda = debug
    pool = torch.randn(8, 2, 16, 16, device="cuda")
    pool0 = pool.clone()
    src, dst = dev(np.array([0, 1, 2], np.int32)), dev(np.array([5, 2, 6], np.int32))  # slot 2 both ways
    with pytest.raises(kda.KdaError) as e:
        kda.kda_state_copy(pool, src, pool, dst)
    assert e.value.code == INVALID_ARG
    with pytest.raises(kda.KdaError):
        kda.kda_state_copy(pool, src, pool, dev(np.array([5, 6, 5], np.int32)))  # a repeated destination
    torch.cuda.synchronize()
    assert torch.equal(pool, pool0)
    # one source feeding two destinations is a valid fork; so is the same ids across two pools
    kda.kda_state_copy(pool, dev(np.array([0, 0], np.int32)), pool, dev(np.array([5, 6], np.int32)))
    other = torch.zeros_like(pool)
    kda.kda_state_copy(pool, src, other, src)
    torch.cuda.synchronize()
    assert torch.equal(pool[5], pool0[0]) and torch.equal(pool[6], pool0[0]) and torch.equal(other[:3], pool0[:3])


def test_debug_mode_rejects_snapshot_into_a_sequence_slot(debug):
    kda = debug
    prob = synth.varlen(seed=39, H=2, d=32, num_slots=8, num_extra=8, snapshot_every_chunks=1, lengths=[130, 70],
                        dtype=synth.F32)
    run = PrefillRun(prob)
    pool0 = run.pool.clone()
    c = run.common()
    # snapshots into the state pool itself, with one extra slot equal to a sequence's own slot
    extra_ids = np.array([[6, 7], [int(prob.slot_ids[0]), 5]], np.int32)
    c.update(extra_pool=run.pool, extra_slot_ids=dev(extra_ids))
    with pytest.raises(kda.KdaError) as e:
        kda.kda_prefill_varlen(*run.args(), workspace=run.varlen_workspace(kda), **c)
    assert e.value.code == INVALID_ARG
    torch.cuda.synchronize()
    assert torch.equal(run.pool, pool0) and status(run.status) == (0, 0)


def test_prep_wait_gives_up_and_flags_timeout(cuda):
    kda = cuda
    prob = synth.varlen(seed=40, H=2, d=128, num_slots=3, num_extra=4, snapshot_every_chunks=0, lengths=[200, 90])
    run = PrefillRun(prob)
    ws = run.varlen_workspace(kda)
    ws.fill_(0x5A)
    pool0, ws0 = run.pool.clone(), ws.clone()
    kda.kda_set_test_fault(kda.KDA_TEST_FAULT_STALL_RECORD_INPUTS)
    try:
        kda.kda_prefill_records(*run.args(), workspace=ws, **run.common())
    finally:
        kda.kda_set_test_fault(kda.KDA_TEST_FAULT_NONE)
    torch.cuda.synchronize()  # the kernel returned: every CTA gave up its wait
    flags, work = status(run.status)
    assert flags == kda.KDA_DEV_TIMEOUT and work == 0
    assert torch.equal(ws, ws0) and torch.equal(run.pool, pool0)  # no record written, no state touched
    # the context is still usable: the same problem, run normally, matches the oracle
    run2 = PrefillRun(prob).run_varlen(kda)
    assert status(run2.status) == (0, prob.T * prob.H)
    ref = oracle_prefill(prob)
    assert rel_err(host(run2.out), ref["o"]) <= 2e-3
