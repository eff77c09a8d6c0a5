"""GPU parity: packed varlen prefill and the segmented (KCP) prefill against the oracle, through the C ABI.

Small cases span several 64-token chunks with ragged tails, empty and one-token sequences, and the
snapshot ping-pong; the full-size workloads (single 8K request, 16-sequence varlen, 1M tokens) follow in
test_gpu_fullsize.py."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests._gpu import (PrefillRun, bf16_bits, dev, expected_extra_pool, host, oracle_prefill, prefix_problem, rel_err,
                        status)

pytestmark = pytest.mark.gpu

TOL = {synth.BF16: 2e-3, synth.F32: 1e-5}


def _check_against_oracle(run: PrefillRun, ref, tol):
    prob = run.prob
    assert rel_err(host(run.out), ref["o"]) <= tol
    got = host(run.pool[run.slots.long()])
    assert rel_err(got, ref["s_final"]) <= tol
    untouched = np.ones(prob.pool.shape[0], bool)
    untouched[prob.slot_ids] = False
    assert np.array_equal(run.pool.cpu().numpy()[untouched], prob.pool[untouched])
    if run.extra is not None and not prob.snapshot_every_chunks:
        assert np.array_equal(run.extra.cpu().numpy(), prob.extra_pool), "no snapshots were requested"
    elif run.extra is not None:
        exp = expected_extra_pool(prob, ref)
        got_extra = host(run.extra)
        assert rel_err(got_extra, exp) <= tol
        written = np.zeros(prob.extra_pool.shape[0], bool)
        for i, s in enumerate(ref["snaps"]):
            for m in range(1, min(len(s), 2) + 1):
                written[prob.extra_slot_ids[i, (len(s) - m) & 1]] = True
        assert np.all(got_extra[~written] == 0), "extra slots without a snapshot must stay untouched"


def test_tiny_fp32(cuda):
    """1 sequence, T = 64, H = 2, d = 16, fp32, zero initial state: all outputs and the final state."""
    prob = synth.tiny()
    run = PrefillRun(prob).run_varlen(cuda)
    ref = oracle_prefill(prob)
    assert status(run.status) == (0, prob.T * prob.H)
    _check_against_oracle(run, ref, TOL[synth.F32])


VARLEN_CASES = [
    # lengths chosen to hit: empty, single token, chunk-1, chunk, chunk+1, several chunks + tail, and
    # snapshot intervals (every 2 chunks = 128 tokens) with odd and even snapshot counts
    dict(d=128, dtype=synth.BF16, lengths=[0, 1, 63, 64, 65, 200, 300, 513], snap=2, H=3),
    dict(d=64, dtype=synth.F32, lengths=[129, 7, 256, 64], snap=1, H=2),
    dict(d=32, dtype=synth.BF16, lengths=[384, 5], snap=3, H=2),
    dict(d=16, dtype=synth.F32, lengths=[1000, 17, 0], snap=4, H=4),
]


def _vid(c):
    return f"d{c['d']}_{'bf16' if c['dtype'] == synth.BF16 else 'f32'}_n{len(c['lengths'])}"


def _varlen(c, seed=31):
    n = len(c["lengths"])
    return synth.varlen(seed=seed, H=c["H"], d=c["d"], num_slots=2 * n + 3, num_extra=2 * n + 5,
                        snapshot_every_chunks=c["snap"], dtype=c["dtype"], lengths=c["lengths"])


@pytest.mark.parametrize("case", VARLEN_CASES, ids=_vid)
def test_varlen_with_snapshots(cuda, case):
    prob = _varlen(case)
    run = PrefillRun(prob).run_varlen(cuda)
    ref = oracle_prefill(prob)
    assert status(run.status) == (0, prob.T * prob.H)
    _check_against_oracle(run, ref, TOL[prob.in_dtype])


@pytest.mark.parametrize("case", VARLEN_CASES, ids=_vid)
@pytest.mark.parametrize("segment_len", [64, 192])
def test_segmented_matches_oracle(cuda, case, segment_len):
    prob = _varlen(case, seed=32)
    run = PrefillRun(prob).run_segmented(cuda, segment_len)
    ref = oracle_prefill(prob)
    assert status(run.status)[0] == 0
    _check_against_oracle(run, ref, TOL[prob.in_dtype])


@pytest.mark.parametrize("path", ["varlen", "segmented"])
def test_decay_floor_uses_block_references(cuda, path):
    """Log-decay at the floor g = -5 in some chunks: their decay span exceeds 80, so the pair decays use
    16-token block references; other chunks keep the single-reference form."""
    prob = synth.varlen(seed=36, H=2, d=128, num_slots=5, num_extra=6, snapshot_every_chunks=1,
                        lengths=[150, 64, 200])
    g = prob.g.copy()
    g[20:100] = -5.0         # spans two chunks of the first sequence
    g[214:230, 1] = -5.0     # one head only, inside the second sequence's chunk
    prob.g = g
    run = PrefillRun(prob)
    run = run.run_varlen(cuda) if path == "varlen" else run.run_segmented(cuda, 128)
    ref = oracle_prefill(prob)
    assert status(run.status)[0] == 0
    _check_against_oracle(run, ref, TOL[synth.BF16])


def test_init_zero_and_bf16_output(cuda):
    prob = synth.varlen(seed=33, H=2, d=128, num_slots=6, num_extra=4, snapshot_every_chunks=0,
                        lengths=[100, 250])
    prob.init_zero = True
    run32 = PrefillRun(prob).run_varlen(cuda)
    ref = oracle_prefill(prob)
    _check_against_oracle(run32, ref, TOL[synth.BF16])
    run16 = PrefillRun(prob, out_dtype=torch.bfloat16).run_varlen(cuda)
    assert np.array_equal(bf16_bits(run16.out), synth.f32_to_bf16(run32.out.cpu().numpy()))
    assert torch.equal(run16.pool, run32.pool)


def test_segment_fragments_and_scan(cuda):
    """Phase outputs of the segmented path: per segment, S~ (zero input state) and the cumulative
    transition M; the scan's entry states equal the oracle's states at the segment boundaries."""
    kda = cuda
    seg = 128
    prob = synth.varlen(seed=34, H=2, d=32, num_slots=4, num_extra=8, snapshot_every_chunks=0,
                        lengths=[300, 128, 70], dtype=synth.F32)
    run = PrefillRun(prob)
    ws = run.workspace_for(kda, seg)
    c = {k: v for k, v in run.common().items()}
    kda.kda_segment_fragments(*run.args(), seg, ws, **c)
    kda.kda_fragment_scan(*run.args(), seg, ws, **c)
    torch.cuda.synchronize()
    N, H, d = prob.N, prob.H, prob.dk
    P = -(-int(prob.lengths.max()) // seg)
    frag_elems = N * P * H * d * 2 * d
    frag_bytes = -(-frag_elems * 4 // 256) * 256
    wsf = ws.view(torch.float32)
    frag = host(wsf[:frag_elems]).reshape(N, P, H, d, 2 * d)
    entry = host(wsf[frag_bytes // 4:frag_bytes // 4 + N * P * H * d * d]).reshape(N, P, H, d, d)
    cu = prob.cu_seqlens.astype(np.int64)
    for i in range(N):
        n_seg = -(-int(prob.lengths[i]) // seg)
        a, b = int(cu[i]), int(cu[i + 1])
        bounds = [p * seg for p in range(n_seg)] + [b - a]  # relative to the sequence start
        sl = lambda x: np.ascontiguousarray(x[a:b])
        M = oracle.transition(sl(prob.k), sl(prob.g), sl(prob.beta), bounds)
        zero = oracle.recurrence(sl(prob.q), sl(prob.k), sl(prob.v), sl(prob.g), sl(prob.beta), bounds, s0=None,
                                 want_o=False)
        for p in range(n_seg - 1):  # the last segment's fragment is not needed and not computed
            # M is a product of seg transitions; fp32 rounding accumulates about seg * 2^-24 relative
            # (~8e-6 rms at 128 tokens), so the intermediate M gets 1e-4.  The 1e-5 bar applies to the
            # states and outputs computed from it (test_segmented_matches_oracle).
            assert rel_err(frag[i, p, :, :, d:], M[p]) <= 1e-4
            assert rel_err(frag[i, p, :, :, :d], zero["s_final"][p]) <= 1e-5
        # entry states: oracle states at the segment starts
        full = oracle.recurrence(prob.q[cu[i]:cu[i + 1]], prob.k[cu[i]:cu[i + 1]], prob.v[cu[i]:cu[i + 1]],
                                 prob.g[cu[i]:cu[i + 1]], prob.beta[cu[i]:cu[i + 1]], [0, int(prob.lengths[i])],
                                 s0=prob.pool[prob.slot_ids[i]][None].astype(np.float64), snap_every=seg,
                                 want_o=False)
        expect = [prob.pool[prob.slot_ids[i]].astype(np.float64)] + list(full["snaps"][0])
        for p in range(n_seg):
            assert rel_err(entry[i, p], expect[p]) <= 1e-5


@pytest.mark.parametrize("dtype,tol", [(synth.F32, 1e-5), (synth.BF16, 2e-3)], ids=["f32", "bf16"])
def test_segment_scan_d128(cuda, dtype, tol):
    """The fragment scan at d = 128 (the tensor-core kernel): every entry state equals the oracle's state
    at that segment's start, for sequences of three, two and one segments (each with a ragged tail).  With
    bf16 inputs the fragments come from the tensor-core chain, whose operand records lead the workspace."""
    kda = cuda
    seg = 128
    prob = synth.varlen(seed=37, H=2, d=128, num_slots=4, num_extra=8, snapshot_every_chunks=0,
                        lengths=[300, 200, 70], dtype=dtype)
    run = PrefillRun(prob)
    ws = run.workspace_for(kda, seg)
    c = {k: v for k, v in run.common().items()}
    rec_bytes = kda.kda_prefill_workspace_size(*run.args(), **{k: v for k, v in c.items() if k != "dev_status"})
    kda.kda_prefill_records(*run.args(), workspace=ws, **c)  # records (nothing on the CUDA-core path)
    kda.kda_segment_fragments(*run.args(), seg, ws, **c)
    kda.kda_fragment_scan(*run.args(), seg, ws, **c)
    torch.cuda.synchronize()
    assert status(run.status)[0] == 0
    N, H, d = prob.N, prob.H, prob.dk
    P = -(-int(prob.lengths.max()) // seg)
    frag_elems = N * P * H * d * 2 * d
    frag_bytes = -(-frag_elems * 4 // 256) * 256
    base = (rec_bytes + frag_bytes) // 4  # workspace: [records][fragments][entry states]
    wsf = ws.view(torch.float32)
    entry = host(wsf[base:base + N * P * H * d * d]).reshape(N, P, H, d, d)
    cu = prob.cu_seqlens.astype(np.int64)
    for i in range(N):
        n_seg = -(-int(prob.lengths[i]) // seg)
        full = oracle.recurrence(prob.q[cu[i]:cu[i + 1]], prob.k[cu[i]:cu[i + 1]], prob.v[cu[i]:cu[i + 1]],
                                 prob.g[cu[i]:cu[i + 1]], prob.beta[cu[i]:cu[i + 1]], [0, int(prob.lengths[i])],
                                 s0=prob.pool[prob.slot_ids[i]][None].astype(np.float64), snap_every=seg,
                                 want_o=False)
        expect = [prob.pool[prob.slot_ids[i]].astype(np.float64)] + list(full["snaps"][0])
        for p in range(n_seg):
            assert rel_err(entry[i, p], expect[p]) <= tol


def test_bad_cu_seqlens_flagged(cuda):
    kda = cuda
    prob = synth.varlen(seed=35, H=2, d=16, num_slots=4, num_extra=4, snapshot_every_chunks=0,
                        lengths=[40, 30], dtype=synth.F32)
    run = PrefillRun(prob)
    run.cu = dev(np.array([0, 50, 40], np.int32))  # decreasing: sequence 1 is invalid
    pool0 = run.pool.clone()
    kda.kda_prefill_varlen(*run.args(), workspace=run.varlen_workspace(kda), **run.common())
    torch.cuda.synchronize()
    flags, work = status(run.status)
    assert flags & kda.KDA_DEV_SEQ_OOB
    assert torch.equal(run.pool[int(prob.slot_ids[1])], pool0[int(prob.slot_ids[1])])


SNAP_EXACT_CASES = [
    # tcgen05 chunk path (bf16, d = 128) and the token-sequential path (fp32 or d < 128); every sequence but
    # one has a length that is a multiple of the snapshot interval, so its last snapshot is its final state
    dict(d=128, dtype=synth.BF16, lengths=[512, 300, 1024, 128], snap=2, H=2),
    dict(d=64, dtype=synth.F32, lengths=[256, 200, 448], snap=1, H=2),
    dict(d=32, dtype=synth.BF16, lengths=[384, 576, 200, 64], snap=3, H=2),
]


@pytest.mark.parametrize("case", SNAP_EXACT_CASES, ids=_vid)
@pytest.mark.parametrize("path", ["varlen", "segmented"])
def test_snapshots_bit_exact(cuda, case, path):
    """Each snapshot the prefill leaves in the ping-pong pool is, bit for bit, the final state of a prefill
    of exactly that prefix (m x interval tokens) on the same path (same segment length); for a sequence
    whose length is a multiple of the interval, the last snapshot equals its final pool state byte for
    byte.  Snapshots are copies of the carried state ("SGLang and Miles: day-0 support for Kimi K3", three
    state movements on the forward stream), so no tolerance applies."""
    seg = 192
    prob = _varlen(case, seed=38)
    full = PrefillRun(prob)
    full = full.run_varlen(cuda) if path == "varlen" else full.run_segmented(cuda, seg)
    assert status(full.status)[0] == 0
    every = case["snap"] * 64
    extra = full.extra.cpu().numpy()
    pool = full.pool.cpu().numpy()
    checked = 0
    for i, n in enumerate(prob.lengths):
        n_snap = int(n) // every
        for m in range(max(1, n_snap - 1), n_snap + 1):  # the two snapshots that survive the call
            pre = PrefillRun(prefix_problem(prob, i, m * every))
            pre = pre.run_varlen(cuda) if path == "varlen" else pre.run_segmented(cuda, seg)
            assert status(pre.status)[0] == 0
            want = pre.pool.cpu().numpy()[prob.slot_ids[i]]
            got = extra[prob.extra_slot_ids[i, (m - 1) & 1]]
            assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), f"seq {i} snapshot {m}"
            checked += 1
        if n_snap and int(n) % every == 0:
            last = extra[prob.extra_slot_ids[i, (n_snap - 1) & 1]]
            assert np.array_equal(last.view(np.uint32), pool[prob.slot_ids[i]].view(np.uint32)), f"seq {i}"
    assert checked == sum(min(int(n) // every, 2) for n in prob.lengths) > 0
