"""The allocation-free segmented prefill (kda_prefill_segmented_noalloc) against the existing entry point.

Callers such as a plugin inside an inference server (which owns all device memory and gives plugins no
allocation hook), or a serving loop that may not call cudaMalloc after start-up, cannot pass a workspace;
this entry point takes its whole workspace (operand records, fragments, entry states) from a fixed
32 MiB array inside the library.  This file is collected
last on purpose: if it fails, a run that stops at the first failure has already run every other test."""
import numpy as np
import pytest
import torch

import synth
from tests._gpu import PrefillRun, status

pytestmark = pytest.mark.gpu

SEGMENT = 256  # one 1024-token sequence, H = 4, d = 128: about 13 MiB of scratch


def test_noalloc_matches_workspace_entry_point_twice(cuda):
    kda = cuda
    prob = synth.prefill_8k(T=1024, H=4)
    ref = PrefillRun(prob).run_segmented(kda, SEGMENT)  # the existing entry point, caller workspace
    assert status(ref.status)[0] == 0
    for call in range(2):  # two calls in a row: the second reuses the array as the first left it
        run = PrefillRun(prob)
        kda.kda_prefill_segmented_noalloc(*run.args(), SEGMENT, **run.common())
        torch.cuda.synchronize()
        assert status(run.status)[0] == 0 and status(run.status)[1] > 0
        # same inputs, same kernels, same launch shapes: only the scratch's address differs, so the results
        # must agree bit for bit (a tolerance could hide bytes left in the shared array by the last call)
        assert torch.equal(run.out, ref.out), f"call {call}: outputs differ"
        assert torch.equal(run.pool, ref.pool), f"call {call}: final state differs"


def test_noalloc_rejects_problems_beyond_its_scratch(cuda):
    kda = cuda
    prob = synth.prefill_8k(T=2048, H=12)
    run = PrefillRun(prob)
    pool0 = run.pool.clone()
    # 2048 tokens x 12 heads: the chunk operand records alone take about 58 MiB > 32 MiB
    with pytest.raises(kda.KdaError) as e:
        kda.kda_prefill_segmented_noalloc(*run.args(), 64, **run.common())
    assert e.value.code == 3  # KDA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.equal(run.pool, pool0) and status(run.status) == (0, 0)
