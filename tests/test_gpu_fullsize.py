"""GPU parity at the full workload sizes, in the launch configurations the benchmark times.

* single-request prefill: B=1, T=8192, H=12, d=128, bf16 q/k/v, S0 ~ N(0, 0.02): every output and the
  final state, through kda_prefill_varlen and kda_prefill_segmented;
* varlen prefill: 16 sequences, lengths log-uniform in [512, 32768], 256-slot pool, snapshots every 4
  chunks: 4096 sampled outputs, every final state and both ping-pong snapshot entries;
* long-context prefill: T = 1,048,576 as 64 segments of 16,384 tokens: 4096 sampled outputs and the
  final state (slow: the fp64 oracle runs the whole recurrence on the host).
"""
import numpy as np
import pytest
import torch

import synth
from tests._gpu import PrefillRun, expected_extra_pool, host, oracle_prefill, prefix_problem, rel_err, status

pytestmark = pytest.mark.gpu

TOL = 2e-3
SEGMENT_8K = 704  # the segment length the benchmark uses for the single 8K request (12 segments)


@pytest.fixture(scope="module")
def p8k():
    prob = synth.prefill_8k()
    return prob, oracle_prefill(prob)


def test_prefill_8k_varlen(cuda, p8k):
    prob, ref = p8k
    run = PrefillRun(prob).run_varlen(cuda)
    assert status(run.status) == (0, prob.T * prob.H)
    assert rel_err(host(run.out), ref["o"]) <= TOL
    assert rel_err(host(run.pool[0]), ref["s_final"][0]) <= TOL


def test_prefill_8k_segmented(cuda, p8k):
    prob, ref = p8k
    run = PrefillRun(prob).run_segmented(cuda, SEGMENT_8K)
    assert status(run.status)[0] == 0
    assert rel_err(host(run.out), ref["o"]) <= TOL
    assert rel_err(host(run.pool[0]), ref["s_final"][0]) <= TOL


def test_varlen_full(cuda):
    prob = synth.varlen()
    samples = np.sort(np.argsort(synth.uniform(prob.seed, synth.S_SAMPLES, prob.T), kind="stable")[:4096])
    ref = oracle_prefill(prob, want_o=False, sample_t=samples)
    run = PrefillRun(prob).run_varlen(cuda)
    assert status(run.status) == (0, prob.T * prob.H)
    out = host(run.out[torch.from_numpy(samples).cuda()])
    assert rel_err(out, ref["o_samples"]) <= TOL
    assert rel_err(host(run.pool[run.slots.long()]), ref["s_final"]) <= TOL
    exp = expected_extra_pool(prob, ref)
    used = np.unique(prob.extra_slot_ids.ravel())
    assert rel_err(host(run.extra)[used], exp[used]) <= TOL
    # the latest snapshot of the longest sequence is, bit for bit, the final state of a prefill of that prefix
    i = int(np.argmax(prob.lengths))
    every = prob.snapshot_every_chunks * 64
    m = int(prob.lengths[i]) // every
    pre = PrefillRun(prefix_problem(prob, i, m * every)).run_varlen(cuda)
    assert status(pre.status)[0] == 0
    want = pre.pool[int(prob.slot_ids[i])]
    assert torch.equal(run.extra[int(prob.extra_slot_ids[i, (m - 1) & 1])], want)


@pytest.mark.slow
def test_long_1m_segmented(cuda):
    prob = synth.long_1m()
    ref = oracle_prefill(prob, want_o=False, sample_t=prob.sample_t)
    run = PrefillRun(prob, out_dtype=torch.float32).run_segmented(cuda, prob.segment_len)
    assert status(run.status)[0] == 0
    out = host(run.out[torch.from_numpy(prob.sample_t).cuda()])
    assert rel_err(out, ref["o_samples"]) <= TOL
    assert rel_err(host(run.pool[0]), ref["s_final"][0]) <= TOL
