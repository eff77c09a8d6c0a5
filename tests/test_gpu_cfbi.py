"""CF-BI: one row-level contract for prefill and decode ("Kimi K3.1 inference zero mismatch", section 6.1).

* Values: outputs and chunk-boundary states against the fp64 oracle recurrence (2e-3 of the rms for bf16
  inputs, 1e-5 for fp32 inputs).
* Bit identity: a sequence prefilled in one call, prefilled in two calls, or prefilled up to any position
  and then decoded token by token gives the same output bits, the same entry state, the same open-chunk
  row cache and the same row count.  A request's decode output does not depend on the batch around it.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests._gpu import dev, host, rel_err, status

pytestmark = pytest.mark.gpu

CH, RF = 16, 420


def _problem(lengths, H, dtype, seed):
    p = synth.varlen(seed=seed, H=H, d=128, lengths=lengths, num_slots=len(lengths) + 3, dtype=dtype)
    return p


def _state(p, torch_dtype_out=torch.float32):
    pool = dev(p.pool).clone()
    cache = torch.zeros(p.pool.shape[0], p.H, CH, RF, dtype=torch.float32, device="cuda")
    counts = torch.zeros(p.pool.shape[0], p.H, dtype=torch.int32, device="cuda")
    return pool, cache, counts


def _tok(p, lo, hi):
    """Token-major input slices [lo, hi) as device tensors."""
    return [dev(np.ascontiguousarray(x[lo:hi])) for x in (p.q, p.k, p.v, p.g, p.beta)]


@pytest.mark.parametrize("dtype,tol", [(synth.BF16, 2e-3), (synth.F32, 1e-5)], ids=["bf16", "f32"])
def test_cfbi_prefill_matches_oracle(cuda, dtype, tol):
    kda = cuda
    lengths = [1, 16, 17, 50, 64]
    p = _problem(lengths, H=2, dtype=dtype, seed=81)
    pool, cache, counts = _state(p)
    q, k, v, g, beta = _tok(p, 0, p.T)
    out = torch.empty(p.T, p.H, 128, dtype=torch.float32, device="cuda")
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    slots = dev(p.slot_ids)
    kda.kda_cfbi_prefill(q, k, v, g, beta, dev(p.cu_seqlens.astype(np.int32)), int(p.lengths.max()), pool, cache,
                         counts, slots, out, dev_status=st)
    torch.cuda.synchronize()
    assert status(st) == (0, p.T * p.H)
    s0 = p.pool[p.slot_ids].astype(np.float64)
    ref = oracle.recurrence(p.q, p.k, p.v, p.g, p.beta, p.cu_seqlens, s0=s0)
    assert rel_err(host(out), ref["o"]) <= tol
    # entry state = the recurrence's state after the last full chunk; counts = the open rows
    cu = p.cu_seqlens
    for i, L in enumerate(lengths):
        full = (L // CH) * CH
        sl = int(p.slot_ids[i])
        assert int(counts[sl, 0]) == L - full and int(counts[sl, 1]) == L - full
        r = oracle.recurrence(*(x[cu[i]:cu[i] + full] for x in (p.q, p.k, p.v, p.g, p.beta)), [0, full],
                              s0=s0[i:i + 1]) if full else {"s_final": s0[i:i + 1]}
        assert rel_err(host(pool[sl]), r["s_final"][0]) <= tol


@pytest.mark.parametrize("split", [0, 7, 16, 33, 49])
def test_prefill_then_decode_is_bit_identical(cuda, split):
    kda = cuda
    T = 50
    p = _problem([T], H=2, dtype=synth.BF16, seed=82)
    cu_all = dev(np.array([0, T], np.int32))
    slots = dev(p.slot_ids)
    # one prefill call over the whole sequence
    pool_a, cache_a, counts_a = _state(p)
    out_a = torch.empty(T, p.H, 128, dtype=torch.bfloat16, device="cuda")
    kda.kda_cfbi_prefill(*_tok(p, 0, T), cu_all, T, pool_a, cache_a, counts_a, slots, out_a)
    # prefill the first `split` tokens, then decode the rest one token at a time
    pool_b, cache_b, counts_b = _state(p)
    out_b = torch.empty(T, p.H, 128, dtype=torch.bfloat16, device="cuda")
    if split:
        kda.kda_cfbi_prefill(*_tok(p, 0, split), dev(np.array([0, split], np.int32)), split, pool_b, cache_b,
                             counts_b, slots, out_b[:split])
    for t in range(split, T):
        o = torch.empty(1, p.H, 128, dtype=torch.bfloat16, device="cuda")
        kda.kda_cfbi_decode(*_tok(p, t, t + 1), pool_b, cache_b, counts_b, slots, o)  # one request: [1, H, .]
        out_b[t] = o[0]
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)
    assert torch.equal(pool_a, pool_b)
    assert torch.equal(counts_a, counts_b)
    sl = int(p.slot_ids[0])
    n = int(counts_a[sl, 0])
    assert torch.equal(cache_a[sl, :, :n], cache_b[sl, :, :n])


def test_two_prefill_calls_are_bit_identical(cuda):
    kda = cuda
    T, cut = 45, 21
    p = _problem([T], H=3, dtype=synth.F32, seed=83)
    slots = dev(p.slot_ids)
    pool_a, cache_a, counts_a = _state(p)
    out_a = torch.empty(T, p.H, 128, device="cuda")
    kda.kda_cfbi_prefill(*_tok(p, 0, T), dev(np.array([0, T], np.int32)), T, pool_a, cache_a, counts_a, slots, out_a)
    pool_b, cache_b, counts_b = _state(p)
    out_b = torch.empty(T, p.H, 128, device="cuda")
    kda.kda_cfbi_prefill(*_tok(p, 0, cut), dev(np.array([0, cut], np.int32)), cut, pool_b, cache_b, counts_b, slots,
                         out_b[:cut])
    kda.kda_cfbi_prefill(*_tok(p, cut, T), dev(np.array([0, T - cut], np.int32)), T - cut, pool_b, cache_b, counts_b,
                         slots, out_b[cut:])
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b) and torch.equal(pool_a, pool_b) and torch.equal(counts_a, counts_b)


@pytest.mark.parametrize("B,H", [(6, 2), (200, 5)], ids=["B6H2", "B200H5"])
def test_decode_is_batch_invariant(cuda, B, H):
    """A request's decode output and state do not depend on which other requests share the batch.  B200H5:
    1000 (request, head) units, two or three per persistent CTA, with every row count (and so the chunk
    fold); the batch also matches the prefill kernel run over the same tokens, bit for bit."""
    kda = cuda
    S = B + 4
    p = synth.decode_verify(seed=84, B=B, W=1, H=H, d=128, num_slots=S)
    rng = np.random.default_rng(0)
    counts0 = torch.from_numpy(rng.integers(0, CH, size=(S, H)).astype(np.int32)).cuda()
    cache0 = torch.from_numpy(rng.standard_normal((S, H, CH, RF)).astype(np.float32) * 0.1).cuda()
    cache0[..., 256:384] = -torch.arange(CH, device="cuda").view(1, 1, CH, 1) * 0.05  # plausible G rows
    pool0 = dev(p.pool)
    ins = [dev(x) for x in (p.q, p.k, p.v, p.g, p.beta)]
    slots = dev(p.slot_ids)
    pool, cache, counts = pool0.clone(), cache0.clone(), counts0.clone()
    out_all = torch.empty(B, H, 128, device="cuda")
    kda.kda_cfbi_decode(*ins, pool, cache, counts, slots, out_all)
    # the same tokens as B one-token sequences through the prefill kernel: the same bits
    pool_p, cache_p, counts_p = pool0.clone(), cache0.clone(), counts0.clone()
    out_p = torch.empty(B, H, 128, device="cuda")
    kda.kda_cfbi_prefill(*ins, dev(np.arange(B + 1, dtype=np.int32)), 1, pool_p, cache_p, counts_p, slots, out_p)
    torch.cuda.synchronize()
    assert torch.equal(out_p, out_all) and torch.equal(pool_p, pool) and torch.equal(counts_p, counts)
    assert torch.equal(cache_p, cache)
    for b in range(B):
        pl, ca, co = pool0.clone(), cache0.clone(), counts0.clone()
        o = torch.empty(1, H, 128, device="cuda")
        kda.kda_cfbi_decode(*(x[b:b + 1].clone() for x in ins), pl, ca, co, slots[b:b + 1].clone(), o)  # fresh, aligned
        torch.cuda.synchronize()
        assert torch.equal(o[0], out_all[b])
        s = int(p.slot_ids[b])
        assert torch.equal(pl[s], pool[s]) and torch.equal(co[s], counts[s]) and torch.equal(ca[s], cache[s])


def test_bad_count_is_flagged(cuda):
    kda = cuda
    p = synth.decode_verify(seed=85, B=2, W=1, H=1, d=128, num_slots=4)
    pool = dev(p.pool)
    cache = torch.zeros(4, 1, CH, RF, device="cuda")
    counts = torch.zeros(4, 1, dtype=torch.int32, device="cuda")
    counts[int(p.slot_ids[1]), 0] = CH  # out of range
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    out = torch.zeros(2, 1, 128, device="cuda")
    kda.kda_cfbi_decode(*(dev(x) for x in (p.q, p.k, p.v, p.g, p.beta)), pool, cache, counts, dev(p.slot_ids), out,
                        dev_status=st)
    torch.cuda.synchronize()
    flags, work = status(st)
    assert flags == kda.KDA_DEV_SLOT_OOB and work == 1
    assert not out[1].any()
