"""KCP across GPUs, the per-rank kernels: three ranks' shards of one sequence run one after another on this
GPU (fragments of every segment of every shard, then the scan over the stacked fragments in token order,
then each shard's outputs from its segments' entry states), as kcp_prefill runs them around its all-gather;
one segment per shard, and three segments per shard at a common segment length.  Outputs, entry states and the final state against the
fp64 oracle's unsplit recurrence (2e-3 of the rms for bf16 inputs, 1e-5 for fp32)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from kda_gated_delta_rule_gb300.kcp import LibraryOps, kcp_segment_len, shard_bounds
from tests._gpu import dev, host, rel_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("per_rank", [1, 3])
@pytest.mark.parametrize("dtype,tol", [(synth.BF16, 2e-3), (synth.F32, 1e-5)], ids=["bf16", "f32"])
def test_three_shards_reproduce_the_unsplit_recurrence(cuda, dtype, tol, per_rank):
    prob = synth.varlen(seed=91, lengths=[500], H=2, num_slots=2, num_extra=2, dtype=dtype)
    T, H = prob.T, prob.H
    s0 = prob.pool[prob.slot_ids[0]]
    b = shard_bounds(T, 3)  # 166, 167, 167 tokens: none a multiple of 64
    seg = kcp_segment_len(T, 3, per_rank) if per_rank > 1 else None  # 64: three segments per shard
    shards = []
    for r in range(3):
        sl = slice(b[r], b[r + 1])
        x = [dev(np.ascontiguousarray(a[sl])) for a in (prob.q, prob.k, prob.v, prob.g, prob.beta)]
        out = torch.empty(b[r + 1] - b[r], H, 128, device="cuda")
        final = torch.empty(H, 128, 128, device="cuda")
        shards.append((LibraryOps(*x, out, final, segment_len=seg), out, final))
    assert all(ops.P == per_rank for ops, _, _ in shards)
    frags = torch.cat([ops.fragments() for ops, _, _ in shards])  # the all-gather's result, in token order
    all_entries = shards[0][0].scan(frags, dev(s0))
    P = per_rank
    for r, (ops, _, _) in enumerate(shards):
        ops.outputs(all_entries[r * P:(r + 1) * P])
    entries = all_entries[::P]
    torch.cuda.synchronize()
    ref = oracle.recurrence(prob.q, prob.k, prob.v, prob.g, prob.beta, [0, T], s0=s0[None].astype(np.float64))
    out = np.concatenate([host(o) for _, o, _ in shards])
    assert rel_err(out, ref["o"]) <= tol
    assert rel_err(host(shards[-1][2]), ref["s_final"][0]) <= tol
    for r in range(1, 3):  # entry state of rank r = the state after the tokens of ranks 0..r-1
        head = oracle.recurrence(*(x[:b[r]] for x in (prob.q, prob.k, prob.v, prob.g, prob.beta)), [0, b[r]],
                                 s0=s0[None].astype(np.float64))
        assert rel_err(host(entries[r]), head["s_final"][0]) <= tol
        assert rel_err(host(shards[r - 1][2]), head["s_final"][0]) <= tol  # each shard's own final state
