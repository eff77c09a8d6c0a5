"""GPU parity: decode step, speculative verify, replay fold and slot copies against the oracle, through the
C ABI.  Full-size workload: 256 requests in a 1024-slot pool, H = 12, d = 128, an 8-token window with
accepted lengths min(Poisson(2.7), 8)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests._gpu import bf16_bits, dev, host, rel_err, status

pytestmark = pytest.mark.gpu

TOL_BF16_IN = 2e-3  # max|d|/rms for bf16 inputs
TOL_F32_IN = 1e-5   # max|d|/rms for the fp32-input path


def _tol(dtype):
    return TOL_BF16_IN if dtype == synth.BF16 else TOL_F32_IN


CASES = [
    dict(B=256, W=8, H=12, d=128, num_slots=1024, dtype=synth.BF16),  # the full decode+verify workload
    dict(B=37, W=5, H=3, d=64, num_slots=50, dtype=synth.F32),
    dict(B=9, W=3, H=2, d=32, num_slots=9, dtype=synth.BF16),
    dict(B=5, W=8, H=2, d=16, num_slots=11, dtype=synth.F32),
]


def _ids(c):
    return f"B{c['B']}_W{c['W']}_H{c['H']}_d{c['d']}_{'bf16' if c['dtype'] == synth.BF16 else 'f32'}"


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_decode_step(cuda, case):
    kda = cuda
    p = synth.decode_verify(B=case["B"], W=case["W"], H=case["H"], d=case["d"], num_slots=case["num_slots"],
                            dtype=case["dtype"])
    q, k, v, g, beta = dev(p.q), dev(p.k), dev(p.v), dev(p.g), dev(p.beta)
    slots = dev(p.slot_ids)
    pool0 = dev(p.pool)
    pool = pool0.clone()
    out = torch.empty(p.B, p.H, p.dv, dtype=torch.float32, device="cuda")
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    kda.kda_decode_step(q, k, v, g, beta, pool, slots, out, dev_status=st)
    torch.cuda.synchronize()
    assert status(st) == (0, p.B * p.H)
    ref_o, ref_s = oracle.decode(p.pool, p.slot_ids, p.q, p.k, p.v, p.g, p.beta)
    assert rel_err(host(out), ref_o) <= _tol(p.in_dtype)
    assert rel_err(host(pool[slots.long()]), ref_s) <= _tol(p.in_dtype)
    untouched = torch.ones(p.pool.shape[0], dtype=torch.bool, device="cuda")
    untouched[slots.long()] = False
    assert torch.equal(pool[untouched], pool0[untouched])
    # bf16 output is the round-to-nearest-even of the fp32 output, bit for bit
    pool2 = pool0.clone()
    out16 = torch.empty(p.B, p.H, p.dv, dtype=torch.bfloat16, device="cuda")
    kda.kda_decode_step(q, k, v, g, beta, pool2, slots, out16)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_bits(out16), synth.f32_to_bf16(out.cpu().numpy()))
    assert torch.equal(pool2, pool)  # deterministic: the same state bits on a repeat


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_verify_and_fold(cuda, case):
    kda = cuda
    p = synth.decode_verify(B=case["B"], W=case["W"], H=case["H"], d=case["d"], num_slots=case["num_slots"],
                            dtype=case["dtype"])
    B, W, H, d = p.B, p.W, p.H, p.dk
    wq, wk, wv, wg, wb = dev(p.wq), dev(p.wk), dev(p.wv), dev(p.wg), dev(p.wbeta)
    slots = dev(p.slot_ids)
    pool0 = dev(p.pool)
    pool = pool0.clone()
    ref_o, ref_states = oracle.verify(p.pool, p.slot_ids, p.wq, p.wk, p.wv, p.wg, p.wbeta)

    # with per-token snapshots: the token-sequential kernel
    out_s = torch.empty(B, W, H, d, dtype=torch.float32, device="cuda")
    rec_s = torch.zeros(kda.kda_replay_bytes(B, W, H, d, d, p.in_dtype), dtype=torch.uint8, device="cuda")
    snaps = torch.empty(B, W, H, d, d, dtype=torch.float32, device="cuda")
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    kda.kda_verify(wq, wk, wv, wg, wb, pool, slots, out_s, rec_s, snapshot_out=snaps, dev_status=st)
    torch.cuda.synchronize()
    assert status(st) == (0, B * H * W)
    assert torch.equal(pool, pool0), "verify must never write the committed state"
    assert rel_err(host(out_s), ref_o) <= _tol(p.in_dtype)
    assert rel_err(host(snaps), ref_states) <= _tol(p.in_dtype)

    # n decode steps from the committed states give the snapshot-after-n states (and outputs) bit for bit
    dpool = pool0.clone()
    dout = torch.empty(B, H, d, dtype=torch.float32, device="cuda")
    for w in range(W):
        kda.kda_decode_step(wq[:, w].contiguous(), wk[:, w].contiguous(), wv[:, w].contiguous(),
                            wg[:, w].contiguous(), wb[:, w].contiguous(), dpool, slots, dout)
        torch.cuda.synchronize()
        assert torch.equal(dpool[slots.long()], snaps[:, w]), f"decode step {w} differs from verify's state"
        assert torch.equal(dout, out_s[:, w])

    # without snapshots (the serving call; the tensor-core kernel for bf16 inputs at d = 128)
    out = torch.empty(B, W, H, d, dtype=torch.float32, device="cuda")
    rec = torch.zeros_like(rec_s)
    st.zero_()
    kda.kda_verify(wq, wk, wv, wg, wb, pool, slots, out, rec, dev_status=st)
    torch.cuda.synchronize()
    assert status(st) == (0, B * H * W)
    assert torch.equal(pool, pool0), "verify must never write the committed state"
    assert rel_err(host(out), ref_o) <= _tol(p.in_dtype)
    assert torch.equal(rec, rec_s)

    # the record holds the exact input bits (k, v, g, beta)
    esz = 2 if p.in_dtype == synth.BF16 else 4
    a256 = lambda x: (x + 255) // 256 * 256
    rows = B * W * H
    raw = rec.cpu().numpy()
    off_v = a256(rows * d * esz)
    off_g = off_v + a256(rows * d * esz)
    off_b = off_g + a256(rows * d * 4)
    assert raw[:rows * d * esz].tobytes() == p.wk.tobytes()
    assert raw[off_v:off_v + rows * d * esz].tobytes() == p.wv.tobytes()
    assert raw[off_g:off_g + rows * d * 4].tobytes() == p.wg.tobytes()
    assert raw[off_b:off_b + rows * 4].tobytes() == p.wbeta.tobytes()

    # fold: commit accepted prefixes
    acc = dev(p.accepted)
    st.zero_()
    kda.kda_verify_replay(pool, slots, rec, acc, W, H, d, d, p.in_dtype, dev_status=st)
    torch.cuda.synchronize()
    assert status(st) == (0, int(p.accepted.sum()) * H)
    for b in range(B):
        n = int(p.accepted[b])
        got = pool[slots[b].long()]
        expect = pool0[slots[b].long()] if n == 0 else snaps[b, n - 1]
        assert torch.equal(got, expect), f"request {b}: fold({n}) is not bit-identical to the recurrence"
    ref_fold = oracle.fold(p.pool, p.slot_ids, p.wq, p.wk, p.wv, p.wg, p.wbeta, p.accepted)
    assert rel_err(host(pool[slots.long()]), ref_fold) <= _tol(p.in_dtype)
    untouched = torch.ones(p.pool.shape[0], dtype=torch.bool, device="cuda")
    untouched[slots.long()] = False
    assert torch.equal(pool[untouched], pool0[untouched])

    # bf16 outputs are the RNE rounding of the fp32 outputs of the same call
    out16 = torch.empty(B, W, H, d, dtype=torch.bfloat16, device="cuda")
    kda.kda_verify(wq, wk, wv, wg, wb, pool0, slots, out16, rec)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_bits(out16), synth.f32_to_bf16(out.cpu().numpy()))


# windows the tensor-core verify takes (W <= 16, padded to 8 or 16 tokens) and one past it
@pytest.mark.parametrize("W", [1, 3, 8, 9, 13, 16, 17])
def test_verify_window_sizes(cuda, W):
    kda = cuda
    p = synth.decode_verify(seed=40 + W, B=19, W=W, H=3, d=128, num_slots=40, dtype=synth.BF16)
    slots = dev(p.slot_ids)
    pool0 = dev(p.pool)
    out = torch.empty(p.B, W, p.H, p.dv, dtype=torch.float32, device="cuda")
    rec = torch.zeros(kda.kda_replay_bytes(p.B, W, p.H, p.dk, p.dv, p.in_dtype), dtype=torch.uint8, device="cuda")
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    kda.kda_verify(dev(p.wq), dev(p.wk), dev(p.wv), dev(p.wg), dev(p.wbeta), pool0, slots, out, rec, dev_status=st)
    torch.cuda.synchronize()
    assert status(st) == (0, p.B * p.H * W)
    ref_o, _ = oracle.verify(p.pool, p.slot_ids, p.wq, p.wk, p.wv, p.wg, p.wbeta)
    assert rel_err(host(out), ref_o) <= TOL_BF16_IN
    assert torch.equal(pool0, dev(p.pool))


def test_verify_steep_gates(cuda):
    """Log-decays of -12 per token: the window's decay spans 192 nats, far beyond fp32's exponent range for
    any single rescaling reference; every factor the verify forms is exp(G_t - G_s) with s <= t."""
    kda = cuda
    p = synth.decode_verify(seed=77, B=6, W=16, H=2, d=128, num_slots=6, dtype=synth.BF16)
    wg = np.full_like(p.wg, -12.0)
    wg[..., ::3] = -0.01  # slow channels keep the state's contribution visible
    slots = dev(p.slot_ids)
    out = torch.empty(p.B, p.W, p.H, p.dv, dtype=torch.float32, device="cuda")
    rec = torch.zeros(kda.kda_replay_bytes(p.B, p.W, p.H, p.dk, p.dv, p.in_dtype), dtype=torch.uint8, device="cuda")
    kda.kda_verify(dev(p.wq), dev(p.wk), dev(p.wv), dev(wg), dev(p.wbeta), dev(p.pool), slots, out, rec)
    torch.cuda.synchronize()
    ref_o, _ = oracle.verify(p.pool, p.slot_ids, p.wq, p.wk, p.wv, wg, p.wbeta)
    got = host(out)
    assert np.isfinite(got).all()
    assert rel_err(got, ref_o) <= TOL_BF16_IN


def test_out_of_range_ids_are_flagged_and_skipped(cuda):
    kda = cuda
    p = synth.decode_verify(B=4, W=3, H=2, d=16, num_slots=8, dtype=synth.F32)
    q, k, v, g, beta = dev(p.q), dev(p.k), dev(p.v), dev(p.g), dev(p.beta)
    pool0 = dev(p.pool)
    pool = pool0.clone()
    bad = p.slot_ids.copy()
    bad[2] = 8  # == num_slots
    out = torch.zeros(4, 2, 16, device="cuda")
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    kda.kda_decode_step(q, k, v, g, beta, pool, dev(bad), out, dev_status=st)
    torch.cuda.synchronize()
    flags, work = status(st)
    assert flags == kda.KDA_DEV_SLOT_OOB and work == 3 * 2
    touched = set(bad[[0, 1, 3]].tolist())
    for s in range(8):
        if s not in touched:
            assert torch.equal(pool[s], pool0[s])
    # accepted length out of range: flagged, slot untouched
    W, H, d = p.W, p.H, p.dk
    rec = torch.zeros(kda.kda_replay_bytes(4, W, H, d, d, p.in_dtype), dtype=torch.uint8, device="cuda")
    wout = torch.zeros(4, W, H, d, device="cuda")
    kda.kda_verify(dev(p.wq), dev(p.wk), dev(p.wv), dev(p.wg), dev(p.wbeta), pool0, dev(p.slot_ids), wout, rec)
    pool = pool0.clone()
    st.zero_()
    acc = dev(np.array([1, W + 1, -1, 0], np.int32))
    kda.kda_verify_replay(pool, dev(p.slot_ids), rec, acc, W, H, d, d, p.in_dtype, dev_status=st)
    torch.cuda.synchronize()
    flags, work = status(st)
    assert flags == kda.KDA_DEV_ACCEPT_OOB and work == 1 * H
    for b in (1, 2, 3):
        assert torch.equal(pool[int(p.slot_ids[b])], pool0[int(p.slot_ids[b])])


def test_verify_out_of_range_slot_is_flagged_and_skipped(cuda):
    """A bad slot id in the tensor-core verify: flagged, its outputs and record untouched, the rest correct
    (more (request, head) items than SMs, so persistent CTAs step over the bad item mid-stream)."""
    kda = cuda
    p = synth.decode_verify(seed=61, B=160, W=6, H=2, d=128, num_slots=200, dtype=synth.BF16)
    bad = p.slot_ids.copy()
    bad[[3, 97]] = [200, -1]
    out = torch.zeros(p.B, p.W, p.H, p.dv, dtype=torch.float32, device="cuda")
    rec = torch.zeros(kda.kda_replay_bytes(p.B, p.W, p.H, p.dk, p.dv, p.in_dtype), dtype=torch.uint8, device="cuda")
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    kda.kda_verify(dev(p.wq), dev(p.wk), dev(p.wv), dev(p.wg), dev(p.wbeta), dev(p.pool), dev(bad), out, rec,
                   dev_status=st)
    torch.cuda.synchronize()
    flags, work = status(st)
    assert flags == kda.KDA_DEV_SLOT_OOB and work == (p.B - 2) * p.H * p.W
    good = np.array([b for b in range(p.B) if b not in (3, 97)])
    ref_o, _ = oracle.verify(p.pool, p.slot_ids[good], p.wq[good], p.wk[good], p.wv[good], p.wg[good],
                             p.wbeta[good])
    got = host(out)
    assert rel_err(got[good], ref_o) <= TOL_BF16_IN
    assert not got[[3, 97]].any()
    rows = p.B * p.W * p.H
    kbytes = rec.cpu().numpy()[:rows * p.dk * 2].view(np.uint16).reshape(p.B, p.W, p.H, p.dk)
    assert not kbytes[[3, 97]].any()
    assert np.array_equal(kbytes[good], p.wk[good])


def test_streams_skip_bad_units_mid_stream(cuda):
    """Decode and fold at full width (256 requests x 12 heads: several units per persistent CTA) with bad
    slot ids and bad accepted lengths scattered through the batch: the bad units are flagged and left alone,
    every other unit gets the bits of a call without them (the same kernels on the good requests only)."""
    kda = cuda
    p = synth.decode_verify(seed=62, B=256, W=8, H=12, d=128, num_slots=1024, dtype=synth.BF16)
    B, W, H, d = p.B, p.W, p.H, p.dk
    bad_rows = np.array([0, 5, 77, 130, 255])
    good = np.setdiff1d(np.arange(B), bad_rows)
    bad = p.slot_ids.copy()
    bad[bad_rows] = [1024, -1, 5000, -7, 1024]
    x = [dev(a) for a in (p.q, p.k, p.v, p.g, p.beta)]
    pool0 = dev(p.pool)
    # decode: all requests with the bad slots, against the good requests alone
    pool, st = pool0.clone(), torch.zeros(2, dtype=torch.int32, device="cuda")
    out = torch.zeros(B, H, d, dtype=torch.bfloat16, device="cuda")
    kda.kda_decode_step(*x, pool, dev(bad), out, dev_status=st)
    pool_g = pool0.clone()
    out_g = torch.zeros(len(good), H, d, dtype=torch.bfloat16, device="cuda")
    gi = torch.from_numpy(good).cuda()
    kda.kda_decode_step(*(t[gi].contiguous() for t in x), pool_g, dev(p.slot_ids[good]), out_g)
    torch.cuda.synchronize()
    assert status(st) == (kda.KDA_DEV_SLOT_OOB, len(good) * H)
    assert torch.equal(out[gi], out_g) and not out[torch.from_numpy(bad_rows).cuda()].any()
    assert torch.equal(pool, pool_g)  # bad slots touched nothing; good ones got the same bits
    # fold: bad accepted lengths (and the bad slots) scattered through the batch
    rec = torch.zeros(kda.kda_replay_bytes(B, W, H, d, d, p.in_dtype), dtype=torch.uint8, device="cuda")
    wout = torch.zeros(B, W, H, d, dtype=torch.bfloat16, device="cuda")
    kda.kda_verify(*(dev(a) for a in (p.wq, p.wk, p.wv, p.wg, p.wbeta)), pool0, dev(p.slot_ids), wout, rec)
    acc = p.accepted.copy()
    acc[[10, 200]] = [W + 1, -2]
    skip = np.zeros(B, bool)
    skip[[10, 200]] = True
    skip[bad_rows] = True
    pool, st = pool0.clone(), torch.zeros(2, dtype=torch.int32, device="cuda")
    kda.kda_verify_replay(pool, dev(bad), rec, dev(acc), W, H, d, d, p.in_dtype, dev_status=st)
    acc_g = acc.copy()
    acc_g[skip] = 0  # nothing accepted: the same units left alone
    pool_g = pool0.clone()
    kda.kda_verify_replay(pool_g, dev(p.slot_ids), rec, dev(acc_g), W, H, d, d, p.in_dtype)
    torch.cuda.synchronize()
    flags, work = status(st)
    # a unit with nothing accepted is skipped before its slot is looked at
    expect = kda.KDA_DEV_ACCEPT_OOB | (kda.KDA_DEV_SLOT_OOB if (acc[bad_rows] > 0).any() else 0)
    assert flags == expect
    assert work == int(acc_g.sum()) * H
    assert torch.equal(pool, pool_g)


def test_state_copy(cuda):
    kda = cuda
    H, d = 12, 128
    src = dev(synth.normal(7, 1, (40, H, d, d), std=0.02))
    dst0 = dev(synth.normal(7, 2, (64, H, d, d), std=0.02))
    dst = dst0.clone()
    ss = dev(synth.distinct_slots(7, 3, 16, 40))
    ds = dev(synth.distinct_slots(7, 4, 16, 64))
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    kda.kda_state_copy(src, ss, dst, ds, dev_status=st)
    torch.cuda.synchronize()
    assert status(st) == (0, 16)
    assert torch.equal(dst[ds.long()], src[ss.long()])
    keep = torch.ones(64, dtype=torch.bool, device="cuda")
    keep[ds.long()] = False
    assert torch.equal(dst[keep], dst0[keep])
    # an out-of-range pair is flagged and skipped
    st.zero_()
    dst = dst0.clone()
    bad = ds.clone()
    bad[0] = 64
    kda.kda_state_copy(src, ss, dst, bad, dev_status=st)
    torch.cuda.synchronize()
    assert status(st) == (kda.KDA_DEV_SLOT_OOB, 15)
    assert torch.equal(dst[bad[1:].long()], src[ss[1:].long()])
