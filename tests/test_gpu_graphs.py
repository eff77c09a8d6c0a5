"""CUDA-graph capture of the library's calls: a serving loop records a step once and replays it.

The calls allocate nothing, never synchronise and never read device memory on the host (with the debug
checks off), so a whole step can be captured on a stream and replayed: a segmented prefill step (state
restore + the prefill's four kernels, launched with programmatic dependent launch), a decode / verify /
fold round, and a batch-invariant decode.  Each replay must give the bits of the same calls run eagerly on
the same inputs, and replaying twice must give them again (the restore inside the graph puts the state
back)."""
import numpy as np
import pytest
import torch

import synth
from tests._gpu import PrefillRun, dev, status

pytestmark = pytest.mark.gpu


def _capture(fn):
    """Runs fn once on a side stream (so one-time host work such as function attributes happens outside the
    capture), then records it into a graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_segmented_prefill_step_replays_bit_exact(cuda):
    kda = cuda
    seg = 512
    prob = synth.prefill_8k(T=2048, H=4)
    ref = PrefillRun(prob).run_segmented(kda, seg)
    run = PrefillRun(prob)
    ws = run.workspace_for(kda, seg)
    pool0 = run.pool.clone()

    def step():
        run.pool.copy_(pool0)
        kda.kda_prefill_segmented(*run.args(), seg, ws, **run.common())

    g = _capture(step)
    for _ in range(2):
        run.out.zero_()
        run.pool.fill_(float("nan"))  # overwritten by the restore inside the graph
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(run.out, ref.out) and torch.equal(run.pool, ref.pool)
    assert status(run.status)[0] == 0


def test_decode_verify_fold_round_replays_bit_exact(cuda):
    kda = cuda
    p = synth.decode_verify(seed=41, B=48, W=8, H=4, d=128, num_slots=64)
    B, W, H, d = p.B, p.W, p.H, p.dk

    def tensors():
        t = dict(pool=dev(p.pool), slots=dev(p.slot_ids), acc=dev(p.accepted),
                 x=[dev(a) for a in (p.q, p.k, p.v, p.g, p.beta)], w=[dev(a) for a in (p.wq, p.wk, p.wv, p.wg, p.wbeta)],
                 out=torch.zeros(B, H, d, dtype=torch.bfloat16, device="cuda"),
                 wout=torch.zeros(B, W, H, d, dtype=torch.bfloat16, device="cuda"),
                 rec=torch.zeros(kda.kda_replay_bytes(B, W, H, d, d, p.in_dtype), dtype=torch.uint8, device="cuda"))
        t["pool0"] = t["pool"].clone()
        return t

    def round_(t):
        t["pool"].copy_(t["pool0"])
        kda.kda_decode_step(*t["x"], t["pool"], t["slots"], t["out"])
        kda.kda_verify(*t["w"], t["pool"], t["slots"], t["wout"], t["rec"])
        kda.kda_verify_replay(t["pool"], t["slots"], t["rec"], t["acc"], W, H, d, d, p.in_dtype)

    ref = tensors()
    round_(ref)
    torch.cuda.synchronize()
    t = tensors()
    g = _capture(lambda: round_(t))
    for _ in range(2):
        t["out"].zero_(), t["wout"].zero_(), t["rec"].zero_()
        g.replay()
        torch.cuda.synchronize()
        for key in ("out", "wout", "rec", "pool"):
            assert torch.equal(t[key], ref[key]), key


def test_cfbi_decode_replays_bit_exact(cuda):
    kda = cuda
    CH, RF = kda.CFBI_CHUNK, kda.CFBI_ROW_FLOATS
    p = synth.decode_verify(seed=42, B=40, W=1, H=3, d=128, num_slots=48)
    rng = np.random.default_rng(1)
    counts0 = dev(rng.integers(0, CH, size=(48, p.H)).astype(np.int32))
    cache0 = dev((rng.standard_normal((48, p.H, CH, RF)) * 0.1).astype(np.float32))
    cache0[..., 256:384] = -torch.arange(CH, device="cuda").view(1, 1, CH, 1) * 0.05
    xs = [dev(a) for a in (p.q, p.k, p.v, p.g, p.beta)]
    slots = dev(p.slot_ids)
    pool0 = dev(p.pool)

    def run(pool, cache, counts, out):
        pool.copy_(pool0), cache.copy_(cache0), counts.copy_(counts0)
        kda.kda_cfbi_decode(*xs, pool, cache, counts, slots, out)

    ref = [pool0.clone(), cache0.clone(), counts0.clone(), torch.empty(p.B, p.H, 128, device="cuda")]
    run(*ref)
    torch.cuda.synchronize()
    mine = [pool0.clone(), cache0.clone(), counts0.clone(), torch.zeros(p.B, p.H, 128, device="cuda")]
    g = _capture(lambda: run(*mine))
    for _ in range(2):
        mine[3].zero_()
        g.replay()
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(mine, ref))
