"""Backward (vector-Jacobian product) of the packed prefill against the fp64 oracle's backward.

The loss is L = sum_t <d_out_t, o_t> + sum_i <d_final_i, S_T(i)> with seeded upstream gradients; every
gradient the library returns (dq, dk, dv, dg, dbeta, dS_0) is compared element by element with the oracle's
on the same input bits.  Tolerance: max |difference| <= TOL x rms(oracle) per gradient tensor.  The library
computes in fp32 from exactly widened inputs, except the products that run on the tensor cores with every
fp32 operand split into bf16 hi + lo (hi*hi + hi*lo + lo*hi, relative operand error ~2^-17): the state
products (dO S^T, dU S^T, U dS'^T, dO U^T) for every input type and, with bf16 inputs, the forward and
reverse chunk chains that produce the entry states, U, dS' and dU.  The chains carry that error through up
to 128 chunk steps (a random walk of ~1e-5 per step in the state).  Measured on the 8192-token workload:
fp32 chains 4e-6 to 6e-5 of the rms, tensor-core chains 2.7e-5 (dS_0) to 9.2e-5 (dg, where the gradient is
a small sum of large terms); a wrong term (a dropped product, a wrong decay factor) gives errors of order 1.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests._gpu import PrefillRun, dev, host, rel_err, status

pytestmark = pytest.mark.gpu

TOL = 1e-4
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "ds0")


class BackwardRun:
    """Device buffers of one backward call on a synth.Prefill problem."""

    def __init__(self, kda, prob, d_out, d_final, init_zero=False):
        self.r = PrefillRun(prob)
        T, H, N = prob.T, prob.H, prob.N
        self.d_out = dev(d_out)
        self.d_final = None if d_final is None else dev(d_final)
        self.out = {n: torch.full((T, H, 128), float("nan"), device="cuda") for n in ("dq", "dk", "dv", "dg")}
        self.out["dbeta"] = torch.full((T, H), float("nan"), device="cuda")
        self.out["ds0"] = torch.full((N, H, 128, 128), float("nan"), device="cuda")
        self.ws = torch.empty(max(kda.kda_backward_workspace_size(T, N, H), 16), dtype=torch.uint8, device="cuda")
        self.status = torch.zeros(2, dtype=torch.int32, device="cuda")
        self.init_zero = init_zero

    def run(self, kda):
        r, o = self.r, self.out
        kda.kda_prefill_backward(r.q, r.k, r.v, r.g, r.beta, r.cu, r.max_seqlen, self.d_out, o["dq"], o["dk"],
                                 o["dv"], o["dg"], o["dbeta"], self.ws,
                                 pool=None if self.init_zero else r.pool,
                                 slot_ids=None if self.init_zero else r.slots, d_final=self.d_final,
                                 d_init=o["ds0"], dev_status=self.status)
        torch.cuda.synchronize()
        return {n: host(t) for n, t in o.items()}


def oracle_grads(prob, d_out, d_final, init_zero=False):
    s0 = None if init_zero else prob.pool[prob.slot_ids]
    return oracle.backward(prob.q, prob.k, prob.v, prob.g, prob.beta, prob.cu_seqlens, d_out, s0=s0,
                           ds_final=d_final)


def check(got, ref, tol=TOL, tol_dg=None):
    errs = {n: rel_err(got[n], ref[n]) for n in NAMES}
    bad = {n: e for n, e in errs.items() if not e <= (tol_dg if n == "dg" and tol_dg else tol)}
    assert not bad, f"errors {errs}"
    return errs


@pytest.mark.parametrize("dtype", [synth.BF16, synth.F32], ids=["bf16", "f32"])
def test_backward_matches_oracle(cuda, dtype):
    """Ragged lengths: one token, exactly one chunk, a chunk plus one, several chunks with a tail."""
    prob = synth.varlen(seed=61, lengths=[1, 64, 65, 200], H=2, num_slots=8, num_extra=8, dtype=dtype)
    d_out, d_final = synth.output_grads(prob, 61)
    run = BackwardRun(cuda, prob, d_out, d_final)
    got = run.run(cuda)
    assert status(run.status) == (0, prob.T * prob.H)
    check(got, oracle_grads(prob, d_out, d_final))


def test_backward_zero_initial_state_and_no_final_gradient(cuda):
    prob = synth.varlen(seed=62, lengths=[130, 7], H=3, num_slots=4, num_extra=4)
    d_out, _ = synth.output_grads(prob, 62)
    run = BackwardRun(cuda, prob, d_out, None, init_zero=True)
    got = run.run(cuda)
    check(got, oracle_grads(prob, d_out, None, init_zero=True))


def test_backward_empty_sequences_pass_the_state_gradient_through(cuda):
    prob = synth.varlen(seed=63, lengths=[0, 70, 0], H=2, num_slots=6, num_extra=6)
    d_out, d_final = synth.output_grads(prob, 63)
    got = BackwardRun(cuda, prob, d_out, d_final).run(cuda)
    ref = oracle_grads(prob, d_out, d_final)
    check(got, ref)
    np.testing.assert_array_equal(got["ds0"][0], d_final[0])
    np.testing.assert_array_equal(got["ds0"][2], d_final[2])


def test_backward_steep_gates_take_pairwise_decays(cuda):
    """Gates far below the pages' floor (g ~ -7): a 16-token block spans more than e^80, so the kernels take
    the pair decays one by one there; values still match.  dg is held to 5e-4: the in-chunk cumulative
    log-decay reaches |G| ~ 450, where fp32 spacing is 3e-5, so each pair decay e^(G_t - G_s) carries a
    relative error near 1e-4 (the chunk algebra run in fp64 with only G rounded to fp32 shows 1.2e-4), and
    here the gradients with respect to g are small (rms 5e-5) next to the terms they are summed from."""
    prob = synth.varlen(seed=64, lengths=[150], H=2, num_slots=2, num_extra=2)
    prob.g = (prob.g * 0 - 7.0 + 0.5 * np.cos(np.arange(prob.g.size)).reshape(prob.g.shape)).astype(np.float32)
    d_out, d_final = synth.output_grads(prob, 64)
    got = BackwardRun(cuda, prob, d_out, d_final).run(cuda)
    check(got, oracle_grads(prob, d_out, d_final), tol_dg=5e-4)


def test_backward_steep_block_in_one_head_only(cuda):
    """Steep gates in one block of one (sequence, head) among ordinary ones: with bf16 inputs the forward
    pass runs on the tensor cores for every (sequence, head), and the flagged one alone is recomputed by the
    CUDA-core chain; every gradient of every sequence and head still matches."""
    prob = synth.varlen(seed=66, lengths=[150, 200, 90], H=3, num_slots=8, num_extra=8)
    assert prob.in_dtype == synth.BF16
    t0 = 150 + 100  # sequence 1, tokens 100..129, head 2
    prob.g[t0:t0 + 30, 2, :] = (-7.0 + 0.5 * np.cos(np.arange(30 * prob.g.shape[2]))).reshape(30, -1)
    d_out, d_final = synth.output_grads(prob, 66)
    got = BackwardRun(cuda, prob, d_out, d_final).run(cuda)
    check(got, oracle_grads(prob, d_out, d_final), tol_dg=5e-4)


def test_backward_bad_slot_is_flagged(cuda):
    prob = synth.varlen(seed=65, lengths=[10, 10], H=1, num_slots=4, num_extra=4)
    prob.slot_ids = np.array([1, 99], np.int32)
    d_out, d_final = synth.output_grads(prob, 65)
    run = BackwardRun(cuda, prob, d_out, d_final)
    run.run(cuda)
    assert status(run.status)[0] == cuda.KDA_DEV_SLOT_OOB


def test_backward_8k_workload(cuda):
    """The benchmark's 8192-token, 12-head bf16 workload: every gradient element against the oracle."""
    prob = synth.prefill_8k()
    d_out, d_final = synth.output_grads(prob, 2)
    got = BackwardRun(cuda, prob, d_out, d_final).run(cuda)
    check(got, oracle_grads(prob, d_out, d_final))
