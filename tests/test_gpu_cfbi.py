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


def _chunked(kda, p, lo, hi, cu, max_len, pool, cache, counts, slots, out, st=None):
    """kda_cfbi_prefill_chunked over tokens [lo, hi) of p with its own workspace."""
    N = cu.numel() - 1
    ws = torch.empty(kda.kda_cfbi_prefill_chunked_workspace_size(hi - lo, N, p.H), dtype=torch.uint8, device="cuda")
    kda.kda_cfbi_prefill_chunked(*_tok(p, lo, hi), cu, max_len, pool, cache, counts, slots, out, ws, dev_status=st)


@pytest.mark.parametrize("dtype,out_dtype", [(synth.BF16, torch.bfloat16), (synth.F32, torch.float32),
                                             (synth.BF16, torch.float32)], ids=["bf16", "f32", "bf16_in_f32_out"])
def test_chunked_prefill_is_bit_identical_to_sequential(cuda, dtype, out_dtype):
    """Ragged sequences (1 to 200 tokens, one empty) continuing from open chunks of every length: outputs,
    states, counts and open-chunk rows of the chunk-parallel prefill equal the token-sequential prefill's."""
    kda = cuda
    lengths = [37, 1, 200, 16, 0, 15, 64, 129, 33, 48]
    p = _problem(lengths, H=3, dtype=dtype, seed=86)
    N, T = len(lengths), p.T
    slots = dev(p.slot_ids)
    # open chunks of different lengths: a first token-sequential prefill of a few tokens per sequence
    pre = [3, 0, 15, 7, 1, 14, 0, 9, 12, 5]
    pool0, cache0, counts0 = _state(p)
    pre_tok = np.concatenate([np.arange(p.cu_seqlens[i], p.cu_seqlens[i] + min(pre[i], lengths[i])) for i in range(N)])
    cu_pre = np.concatenate([[0], np.cumsum([min(pre[i], lengths[i]) for i in range(N)])]).astype(np.int32)
    xs = [dev(np.ascontiguousarray(x[pre_tok])) for x in (p.q, p.k, p.v, p.g, p.beta)]
    kda.kda_cfbi_prefill(*xs, dev(cu_pre), 16, pool0, cache0, counts0, slots,
                         torch.empty(len(pre_tok), p.H, 128, dtype=out_dtype, device="cuda"))
    rest = np.concatenate([np.arange(p.cu_seqlens[i] + min(pre[i], lengths[i]), p.cu_seqlens[i + 1]) for i in range(N)])
    cu_rest = np.concatenate([[0], np.cumsum([lengths[i] - min(pre[i], lengths[i]) for i in range(N)])]).astype(np.int32)
    ys = [dev(np.ascontiguousarray(x[rest])) for x in (p.q, p.k, p.v, p.g, p.beta)]
    TR = len(rest)
    st_a = torch.zeros(2, dtype=torch.int32, device="cuda")
    st_b = torch.zeros(2, dtype=torch.int32, device="cuda")
    pool_a, cache_a, counts_a = pool0.clone(), cache0.clone(), counts0.clone()
    out_a = torch.empty(TR, p.H, 128, dtype=out_dtype, device="cuda")
    kda.kda_cfbi_prefill(*ys, dev(cu_rest), 200, pool_a, cache_a, counts_a, slots, out_a, dev_status=st_a)
    pool_b, cache_b, counts_b = pool0.clone(), cache0.clone(), counts0.clone()
    out_b = torch.empty(TR, p.H, 128, dtype=out_dtype, device="cuda")
    ws = torch.empty(kda.kda_cfbi_prefill_chunked_workspace_size(TR, N, p.H), dtype=torch.uint8, device="cuda")
    kda.kda_cfbi_prefill_chunked(*ys, dev(cu_rest), 200, pool_b, cache_b, counts_b, slots, out_b, ws, dev_status=st_b)
    torch.cuda.synchronize()
    assert status(st_b) == status(st_a) == (0, TR * p.H)
    assert torch.equal(out_a, out_b)
    assert torch.equal(pool_a, pool_b)
    assert torch.equal(counts_a, counts_b)
    for i in range(N):
        sl = int(p.slot_ids[i])
        for h in range(p.H):
            n = int(counts_a[sl, h])
            assert torch.equal(cache_a[sl, h, :n], cache_b[sl, h, :n])
    # and against the fp64 recurrence at the chunk-boundary states (values, not bits)
    tol = 2e-3 if dtype == synth.BF16 else 1e-5
    s0 = p.pool[p.slot_ids].astype(np.float64)
    for i in (2, 7):
        full = (lengths[i] // CH) * CH
        r = oracle.recurrence(*(x[p.cu_seqlens[i]:p.cu_seqlens[i] + full] for x in (p.q, p.k, p.v, p.g, p.beta)),
                              [0, full], s0=s0[i:i + 1])
        assert rel_err(host(pool_b[int(p.slot_ids[i])]), r["s_final"][0]) <= tol


@pytest.mark.parametrize("split", [0, 5, 16, 41])
def test_chunked_prefill_then_decode_is_bit_identical(cuda, split):
    """A sequence prefilled by the chunk-parallel kernels up to `split` and decoded after it gives the bits of
    one token-sequential prefill over the whole sequence."""
    kda = cuda
    T = 60
    p = _problem([T], H=2, dtype=synth.BF16, seed=87)
    slots = dev(p.slot_ids)
    pool_a, cache_a, counts_a = _state(p)
    out_a = torch.empty(T, p.H, 128, dtype=torch.bfloat16, device="cuda")
    kda.kda_cfbi_prefill(*_tok(p, 0, T), dev(np.array([0, T], np.int32)), T, pool_a, cache_a, counts_a, slots, out_a)
    pool_b, cache_b, counts_b = _state(p)
    out_b = torch.empty(T, p.H, 128, dtype=torch.bfloat16, device="cuda")
    if split:
        _chunked(kda, p, 0, split, dev(np.array([0, split], np.int32)), split, pool_b, cache_b, counts_b, slots,
                 out_b[:split])
    for t in range(split, T):
        o = torch.empty(1, p.H, 128, dtype=torch.bfloat16, device="cuda")
        kda.kda_cfbi_decode(*_tok(p, t, t + 1), pool_b, cache_b, counts_b, slots, o)
        out_b[t] = o[0]
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b) and torch.equal(pool_a, pool_b) and torch.equal(counts_a, counts_b)
    sl = int(p.slot_ids[0])
    n = int(counts_a[sl, 0])
    assert torch.equal(cache_a[sl, :, :n], cache_b[sl, :, :n])


def test_chunked_prefill_long_sequence(cuda):
    """3000 tokens in one sequence (188 chunks) and a short one: bits equal to the token-sequential prefill."""
    kda = cuda
    p = _problem([3000, 21], H=2, dtype=synth.BF16, seed=88)
    slots = dev(p.slot_ids)
    cu = dev(p.cu_seqlens.astype(np.int32))
    pool_a, cache_a, counts_a = _state(p)
    out_a = torch.empty(p.T, p.H, 128, dtype=torch.bfloat16, device="cuda")
    kda.kda_cfbi_prefill(*_tok(p, 0, p.T), cu, 3000, pool_a, cache_a, counts_a, slots, out_a)
    pool_b, cache_b, counts_b = _state(p)
    out_b = torch.empty(p.T, p.H, 128, dtype=torch.bfloat16, device="cuda")
    _chunked(kda, p, 0, p.T, cu, 3000, pool_b, cache_b, counts_b, slots, out_b)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b) and torch.equal(pool_a, pool_b) and torch.equal(counts_a, counts_b)


def test_chunked_prefill_errors(cuda):
    """A short workspace is refused before any launch; a bad slot or row count is flagged and that sequence
    left untouched; a sequence longer than max_seqlen is flagged."""
    kda = cuda
    p = _problem([20, 30], H=1, dtype=synth.F32, seed=89)
    slots = dev(p.slot_ids)
    cu = dev(p.cu_seqlens.astype(np.int32))
    pool, cache, counts = _state(p)
    out = torch.zeros(p.T, 1, 128, device="cuda")
    need = kda.kda_cfbi_prefill_chunked_workspace_size(p.T, 2, 1)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(kda.KdaError):
        kda.kda_cfbi_prefill_chunked(*_tok(p, 0, p.T), cu, 30, pool, cache, counts, slots, out, small)
    # sequence 1's row count out of range
    counts[int(p.slot_ids[1]), 0] = CH
    pool0 = pool.clone()
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    _chunked(kda, p, 0, p.T, cu, 30, pool, cache, counts, slots, out, st)
    torch.cuda.synchronize()
    flags, work = status(st)
    assert flags == kda.KDA_DEV_SLOT_OOB and work == 20
    assert torch.equal(pool[int(p.slot_ids[1])], pool0[int(p.slot_ids[1])])
    assert not out[20:].any()
    # max_seqlen below the longest sequence
    counts[int(p.slot_ids[1]), 0] = 0
    st.zero_()
    _chunked(kda, p, 0, p.T, cu, 25, pool, cache, counts, slots, out, st)
    torch.cuda.synchronize()
    assert status(st)[0] == kda.KDA_DEV_SEQ_OOB
