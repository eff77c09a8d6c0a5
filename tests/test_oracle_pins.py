"""Pins for the fp64 oracle: closed forms, invariants, the pages' worked example and brute force.

Each ``check_*`` raises AssertionError when the oracle (optionally with a planted
mistake) disagrees with what the pages and the mathematics fix.  The last test
plants each mistake in the oracle and requires at least one pin to catch it.
"""
import math
import os

import numpy as np
import pytest

import oracle
from tests._bruteforce import chunked, closed_form_states

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example_2d.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            key, val = (s.strip() for s in line.split("="))
            vals[key] = float(val)
    return vals


def _unit_rows(rng, shape):
    x = rng.standard_normal(shape)
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _problem(rng, T, H, dk, dv, g_scale=0.3):
    q = _unit_rows(rng, (T, H, dk))
    k = _unit_rows(rng, (T, H, dk))
    v = rng.standard_normal((T, H, dv))
    g = -np.abs(rng.standard_normal((T, H, dk))) * g_scale
    beta = rng.uniform(0.05, 0.95, (T, H))
    return q, k, v, g, beta


def _run(q, k, v, g, beta, s0=None, mut="none", **kw):
    T = q.shape[0]
    return oracle.recurrence(q, k, v, g, beta, [0, T], s0=None if s0 is None else s0[None], mutation=mut, **kw)


# ---------------------------------------------------------------- pins

def check_beta_zero_pure_decay(mut="none"):
    """beta = 0: S_T = Diag(prod_t alpha_t) S_0, row j scaled by channel j's decays (KDA math box)."""
    rng = np.random.default_rng(11)
    T, H, dk, dv = 9, 2, 6, 5
    q, k, v, g, _ = _problem(rng, T, H, dk, dv)
    beta = np.zeros((T, H))
    s0 = rng.standard_normal((H, dk, dv))
    r = _run(q, k, v, g, beta, s0, mut)
    expect = np.exp(g.sum(axis=0))[:, :, None] * s0
    np.testing.assert_allclose(r["s_final"][0], expect, rtol=1e-13, atol=0)
    # and every output reads the decayed state: o_t = (Diag(prod_{u<=t} alpha_u) S0)^T q_t
    G = np.cumsum(g, axis=0)
    o = np.einsum("thj,hjc->thc", q * np.exp(G), s0)
    np.testing.assert_allclose(r["o"], o, rtol=1e-12, atol=1e-14)


def check_identity_gate_no_write(mut="none"):
    """alpha = 1, beta = 0: the state never changes and o_t = S_0^T q_t."""
    rng = np.random.default_rng(12)
    T, H, dk, dv = 7, 1, 5, 4
    q, k, v, _, _ = _problem(rng, T, H, dk, dv)
    g = np.zeros((T, H, dk))
    beta = np.zeros((T, H))
    s0 = rng.standard_normal((H, dk, dv))
    r = _run(q, k, v, g, beta, s0, mut)
    assert np.array_equal(r["s_final"][0], s0)
    np.testing.assert_allclose(r["o"], np.einsum("thj,hjc->thc", q, s0), rtol=1e-13, atol=1e-15)


def check_naive_linear_attention(mut="none"):
    """alpha = 1, S_0 = 0, distinct standard-basis keys: S_T = sum_t beta_t k_t v_t^T exactly
    (naive linear attention S = sum k v^T on (k, beta v); linear-attention section and the KCP
    reading's section 4.1, where plain linear attention is additive)."""
    rng = np.random.default_rng(13)
    T, H, dk, dv = 6, 2, 8, 3
    q = _unit_rows(rng, (T, H, dk))
    k = np.zeros((T, H, dk))
    for h in range(H):
        for t, j in enumerate(rng.permutation(dk)[:T]):
            k[t, h, j] = 1.0
    v = rng.standard_normal((T, H, dv))
    g = np.zeros((T, H, dk))
    beta = rng.uniform(0.1, 0.9, (T, H))
    r = _run(q, k, v, g, beta, None, mut)
    expect = np.einsum("th,thj,thc->hjc", beta, k, v)
    assert np.array_equal(r["s_final"][0], expect)
    # outputs: o_t = sum_{s<=t} (k_s . q_t) beta_s v_s
    o = np.stack([np.einsum("sh,shj,hj,shc->hc", beta[:t + 1], k[:t + 1], q[t], v[:t + 1]) for t in range(T)])
    np.testing.assert_allclose(r["o"], o, rtol=1e-13, atol=1e-15)


def check_readback_identity(mut="none"):
    """Unit key, any alpha: S_t^T k_t = (1 - beta_t) r_old + beta_t v_t with r_old = (Diag(alpha_t) S_{t-1})^T k_t
    (KDA math box; DeltaNet section for alpha = 1)."""
    rng = np.random.default_rng(14)
    T, H, dk, dv = 12, 2, 8, 5
    _, k, v, g, beta = _problem(rng, T, H, dk, dv, g_scale=0.5)
    s0 = rng.standard_normal((H, dk, dv))
    r = _run(k, k, v, g, beta, s0, mut, snap_every=1)  # q = k reads back along the written key
    states = np.concatenate([s0[None], r["snaps"][0]])
    for t in range(T):
        gated = np.exp(g[t])[:, :, None] * states[t]
        r_old = np.einsum("hjc,hj->hc", gated, k[t])
        expect = (1 - beta[t])[:, None] * r_old + beta[t][:, None] * v[t]
        np.testing.assert_allclose(r["o"][t], expect, rtol=1e-12, atol=1e-12)


def check_worked_example(mut="none"):
    """The pages' 2-D example (tests/golden/worked_example_2d.txt)."""
    gold = _golden()
    s2 = 1 / math.sqrt(2)
    ka, kb = np.array([s2, s2]), np.array([s2, -s2])
    # naive accumulation (reference value only; not KDA): S = 1 k_a^T + 4 k_a^T, read with k_a
    naive = (np.outer(ka, [1.0]) + np.outer(ka, [4.0])).T @ ka
    assert abs(naive[0] - gold["naive_read_a_after_1_then_4"]) < 1e-12

    def run(keys, vals, g, beta, read):
        T = len(keys)
        kk = np.array(keys)[:, None, :]
        vv = np.array(vals, np.float64)[:, None, None]
        gg = np.array(g, np.float64)[:, None, :]
        bb = np.array(beta, np.float64)[:, None]
        qq = np.repeat(np.array(read)[None, None, :], T, axis=0)
        return _run(qq, kk, vv, gg, bb, None, mut)["o"][-1, 0, 0]

    # DeltaNet (alpha = 1), beta = 1: A=1, B=1, A=4
    seq = [ka, kb, ka]
    vals = [1.0, 1.0, 4.0]
    assert abs(run(seq, vals, [[0, 0]] * 3, [1, 1, 1], ka) - gold["deltanet_beta1_read_a"]) < 1e-12
    assert abs(run(seq, vals, [[0, 0]] * 3, [1, 1, 1], kb) - gold["deltanet_beta1_read_b"]) < 1e-12
    # KDA with arbitrary per-channel gates, beta = 1: the last write along k_a reaches the target 4
    for a1, a2 in [(0.3, 0.9), (0.05, 0.6), (1.0, 0.2)]:
        g = [[math.log(a1), math.log(a2)]] * 3
        assert abs(run(seq, vals, g, [1, 1, 1], ka) - gold["kda_beta1_read_a_any_alpha"]) < 1e-12


def check_crosstalk(mut="none"):
    """S = k_a v_a^T + k_b v_b^T read with q = k_a gives v_a + cos(theta) v_b (DeltaNet math box).
    Built as the initial state, with alpha = 1 and beta = 0 so one step only reads.  dv = 3 with
    distinct values, so a transposed read-out is caught."""
    gold = _golden()
    for theta, key in [(math.pi / 3, "crosstalk_read_a_cos_theta_0.5"), (math.pi / 2, "crosstalk_read_a_orthogonal")]:
        ka = np.array([1.0, 0.0, 0.0])
        kb = np.array([math.cos(theta), math.sin(theta), 0.0])
        va, vb = np.array([1.0, -2.0, 0.5]), np.array([1.0, 3.0, -1.0])
        s0 = (np.outer(ka, va) + np.outer(kb, vb))[None]
        r = _run(ka[None, None], ka[None, None], np.zeros((1, 1, 3)), np.zeros((1, 1, 3)), np.zeros((1, 1)), s0, mut)
        np.testing.assert_allclose(r["o"][0, 0], va + math.cos(theta) * vb, rtol=0, atol=1e-14)
        assert abs(r["o"][0, 0, 0] - gold[key]) < 1e-14


def check_bruteforce(mut="none"):
    """T <= 8, explicit dk x dk transition products (unrolled form in the KDA math box) vs the recurrence."""
    rng = np.random.default_rng(15)
    for T, dk, dv in [(1, 3, 2), (4, 5, 3), (8, 6, 4), (8, 4, 7)]:
        q, k, v, g, beta = _problem(rng, T, 1, dk, dv, g_scale=0.6)
        k = k * rng.uniform(0.5, 1.5, (T, 1, 1))  # not unit: the form holds for any k
        s0 = rng.standard_normal((1, dk, dv))
        r = _run(q, k, v, g, beta, s0, mut)
        states = closed_form_states(k[:, 0], v[:, 0], g[:, 0], beta[:, 0], s0[0])
        np.testing.assert_allclose(r["s_final"][0, 0], states[-1], rtol=1e-12, atol=1e-12)
        o = np.einsum("tjc,tj->tc", states, q[:, 0])
        np.testing.assert_allclose(r["o"][:, 0], o, rtol=1e-12, atol=1e-12)


def check_kcp_composition(mut="none"):
    """Segment fragments (M, S~ from a zero input state) compose as S_in2 = M1 S_in1 + S~1 and reproduce
    the unsplit run, for 2, 3 and 5 pieces ("Kimi K3 infra report reading", sections 4.1-4.2)."""
    rng = np.random.default_rng(16)
    T, H, dk, dv = 96, 2, 6, 4
    q, k, v, g, beta = _problem(rng, T, H, dk, dv)
    s0 = rng.standard_normal((H, dk, dv))
    full = _run(q, k, v, g, beta, s0, mut)
    for pieces in (2, 3, 5):
        cuts = np.sort(rng.choice(np.arange(1, T), pieces - 1, replace=False))
        bounds = np.concatenate([[0], cuts, [T]])
        M = oracle.transition(k, g, beta, bounds)
        seg = oracle.recurrence(q, k, v, g, beta, bounds, s0=None, mutation=mut)  # zero-input S~ per segment
        S = s0.copy()
        outs = []
        for p in range(pieces):
            # outputs of segment p from its exact entry state
            a, b = bounds[p], bounds[p + 1]
            rp = oracle.recurrence(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b], [0, b - a], s0=S[None], mutation=mut)
            outs.append(rp["o"])
            S = np.einsum("hij,hjc->hic", M[p], S) + seg["s_final"][p]
        np.testing.assert_allclose(S, full["s_final"][0], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(np.concatenate(outs), full["o"], rtol=1e-11, atol=1e-12)


def check_transition_bruteforce(mut="none"):
    """oracle.transition equals the explicit product of (I - beta k k^T) Diag(alpha) matrices, and is a
    contraction (spectral norm <= 1) for unit keys, beta in (0,1), alpha <= 1."""
    rng = np.random.default_rng(17)
    T, H, dk = 8, 2, 5
    _, k, _, g, beta = _problem(rng, T, H, dk, 1)
    M = oracle.transition(k, g, beta, [0, 3, T])
    from tests._bruteforce import token_transition
    for h in range(H):
        for s, (a, b) in enumerate([(0, 3), (3, T)]):
            P = np.eye(dk)
            for t in range(a, b):
                P = token_transition(k[t, h], g[t, h], beta[t, h]) @ P
            np.testing.assert_allclose(M[s, h], P, rtol=1e-13, atol=1e-14)
            assert np.linalg.norm(M[s, h], 2) <= 1 + 1e-12


def check_column_independence(mut="none"):
    """Column c of S evolves with column c of v alone: per-column runs equal the joint run bit for bit."""
    rng = np.random.default_rng(18)
    T, H, dk, dv = 20, 2, 7, 37  # dv spans several of the oracle's column blocks
    q, k, v, g, beta = _problem(rng, T, H, dk, dv)
    s0 = rng.standard_normal((H, dk, dv))
    joint = _run(q, k, v, g, beta, s0, mut)
    for c in (0, 15, 16, 36):
        one = _run(q, k, np.ascontiguousarray(v[:, :, c:c + 1]), g, beta, np.ascontiguousarray(s0[:, :, c:c + 1]), mut)
        assert np.array_equal(one["s_final"][0, :, :, 0], joint["s_final"][0, :, :, c])
        assert np.array_equal(one["o"][:, :, 0], joint["o"][:, :, c])


def check_chunked_second_formulation(mut="none"):
    """The chunk-parallel UT/WY form (tests/_bruteforce.chunked) equals the sequential oracle to 1e-11,
    over several chunks with a ragged tail, including the strongest decay the pages allow (g = -5)."""
    rng = np.random.default_rng(19)
    T, dk, dv = 150, 16, 8
    for g_mode in ("typical", "floor"):
        q, k, v, g, beta = _problem(rng, T, 1, dk, dv)
        if g_mode == "floor":
            g = np.full_like(g, -5.0)
        s0 = rng.standard_normal((1, dk, dv)) * 0.1
        r = _run(q, k, v, g, beta, s0, mut)
        O, S = chunked(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], s0[0], C=64, L=16)
        scale = np.sqrt(np.mean(r["o"] ** 2))
        assert np.max(np.abs(O - r["o"][:, 0])) <= 1e-11 * max(scale, 1e-300)
        np.testing.assert_allclose(S, r["s_final"][0, 0], rtol=1e-10, atol=1e-12)


PINS = [
    check_beta_zero_pure_decay,
    check_identity_gate_no_write,
    check_naive_linear_attention,
    check_readback_identity,
    check_worked_example,
    check_crosstalk,
    check_bruteforce,
    check_kcp_composition,
    check_transition_bruteforce,
    check_column_independence,
    check_chunked_second_formulation,
]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_chunked_form_finite_in_fp32_at_decay_floor():
    """With every log-decay at the floor -5, the per-block rescaling keeps every factor finite in fp32
    (no factor above exp(16*5)); the fp32 result stays close to the fp64 oracle."""
    rng = np.random.default_rng(20)
    T, dk, dv = 128, 32, 16
    q, k, v, _, beta = _problem(rng, T, 1, dk, dv)
    g = np.full((T, 1, dk), -5.0)
    s0 = rng.standard_normal((1, dk, dv)) * 0.02
    r = _run(q, k, v, g, beta, s0)
    O, S = chunked(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], s0[0], dtype=np.float32)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(S))
    scale = np.sqrt(np.mean(r["o"] ** 2))
    assert np.max(np.abs(O - r["o"][:, 0])) <= 1e-4 * scale


def test_sizes_from_the_pages():
    """64 KB fp32 state per head at K = V = 128 (ReplaySSM section); ~54 MB per request per GPU
    = 12 heads (one TP8 slice of 96) x 69 KDA layers (hybrid KDA memory section)."""
    per_head = 128 * 128 * 4
    assert per_head == 64 * 1024
    per_request = 12 * per_head * 69
    assert abs(per_request / 1e6 - 54.26) < 0.01


def test_oracle_decode_verify_fold_consistent():
    """verify leaves the committed state alone; fold(n) equals the verify state after n tokens; fold(0) is
    the committed state (ReplaySSM section)."""
    rng = np.random.default_rng(21)
    B, W, H, d, slots = 5, 4, 2, 6, 9
    pool = rng.standard_normal((slots, H, d, d))
    pool_copy = pool.copy()
    sid = np.array([3, 0, 8, 5, 1])
    wq = _unit_rows(rng, (B, W, H, d))
    wk = _unit_rows(rng, (B, W, H, d))
    wv = rng.standard_normal((B, W, H, d))
    wg = -np.abs(rng.standard_normal((B, W, H, d))) * 0.3
    wb = rng.uniform(0.1, 0.9, (B, W, H))
    o, states = oracle.verify(pool, sid, wq, wk, wv, wg, wb)
    assert np.array_equal(pool, pool_copy)
    acc = np.array([0, 1, 4, 2, 3])
    f = oracle.fold(pool, sid, wq, wk, wv, wg, wb, acc)
    for b in range(B):
        expect = pool[sid[b]] if acc[b] == 0 else states[b, acc[b] - 1]
        assert np.array_equal(f[b], expect)
    # one decode step = the first window token
    o1, s1 = oracle.decode(pool, sid, wq[:, 0], wk[:, 0], wv[:, 0], wg[:, 0], wb[:, 0])
    assert np.array_equal(s1, states[:, 0])
    assert np.array_equal(o1, o[:, 0])


@pytest.mark.parametrize("mut", [m for m in oracle.MUTATIONS if m != "none"])
def test_planted_mistakes_are_caught(mut):
    """Each planted mistake in the oracle makes at least one pin fail."""
    failed = []
    for pin in PINS:
        if mut == "transposed_read" and pin is not check_crosstalk:
            continue  # the transposed read-out only exists for square single-block states
        try:
            pin(mut)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake '{mut}'"


# ---------------------------------------------------------------- packing, snapshot and sampling bookkeeping
#
# The varlen contract ("SGLang and Miles: day-0 support for Kimi K3", hybrid KDA memory section: every
# sequence has its own slot; snapshots at fixed token boundaries of each sequence) fixes these by
# construction: a packed run is N independent runs, snapshot m of a sequence is its state after m x every
# of its own tokens, and a sampled output is the same output computed in full.  Each test compares two
# different outputs of the oracle (packed vs separate runs, snapshot vs final state, sample vs full), so a
# slip in the offsets (a state carried across a sequence boundary, boundaries counted on packed positions,
# an off-by-one in the sample index) fails one of them.

VARLEN = [300, 64, 0, 530, 63, 1]


def _varlen_problem(seed, H=2, dk=8, dv=8):
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(VARLEN)]).astype(np.int64)
    q, k, v, g, beta = _problem(rng, int(cu[-1]), H, dk, dv)
    s0 = rng.standard_normal((len(VARLEN), H, dk, dv)) * 0.1
    return cu, (q, k, v, g, beta), s0


def test_packed_sequences_are_independent_runs():
    cu, x, s0 = _varlen_problem(51)
    r = oracle.recurrence(*x, cu, s0=s0)
    for i in range(len(VARLEN)):
        sl = slice(cu[i], cu[i + 1])
        alone = oracle.recurrence(*(a[sl] for a in x), [0, VARLEN[i]], s0=s0[i:i + 1])
        np.testing.assert_array_equal(r["o"][sl], alone["o"])
        np.testing.assert_array_equal(r["s_final"][i], alone["s_final"][0])
    # an empty sequence hands its initial state back unchanged
    np.testing.assert_array_equal(r["s_final"][VARLEN.index(0)], s0[VARLEN.index(0)])


@pytest.mark.parametrize("every", [1, 64, 256])
def test_snapshots_count_from_each_sequence_start(every):
    cu, x, s0 = _varlen_problem(52)
    r = oracle.recurrence(*x, cu, s0=s0, snap_every=every)
    for i, L in enumerate(VARLEN):
        snaps = r["snaps"][i]
        assert snaps.shape[0] == L // every
        for m in range(1, L // every + 1):
            sl = slice(cu[i], cu[i] + m * every)
            prefix = oracle.recurrence(*(a[sl] for a in x), [0, m * every], s0=s0[i:i + 1], want_o=False)
            np.testing.assert_array_equal(snaps[m - 1], prefix["s_final"][0])


def test_sampled_outputs_equal_the_full_outputs():
    cu, x, s0 = _varlen_problem(53)
    T = int(cu[-1])
    sample = np.array([0, 1, 299, 300, 363, 364, 893, T - 1], np.int64)
    full = oracle.recurrence(*x, cu, s0=s0)
    part = oracle.recurrence(*x, cu, s0=s0, want_o=False, sample_t=sample)
    np.testing.assert_array_equal(part["o_samples"], full["o"][sample])
    np.testing.assert_array_equal(part["s_final"], full["s_final"])
