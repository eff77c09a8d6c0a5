"""Pins for the fp64 oracle's backward (the vector-Jacobian product of the recurrence).

The backward is fixed by the forward it differentiates, and the forward is pinned by its own tests, so:

* finite differences of the forward oracle along random directions, one input at a time, must equal the
  inner product of the oracle's gradient with the direction (central differences in fp64: agreement to
  about 1e-9 relative, far below any plausible mistake);
* the loss is linear in q (o_t = S_t^T q_t, S_T does not depend on q), so <dq, q> = sum_t <dO_t, o_t>;
  and jointly linear in (v, S_0), so <dv, v> + <dS_0, S_0> = L, both exactly up to rounding;
* with beta = 0 the state only decays, S_t = Diag(prod_{u<=t} alpha_u) S_0, and every gradient has a
  closed form written out here from that product (dk = dv = 0; dq, dS_0, dg, dbeta explicit);
* the chunk-parallel backward algebra (a second formulation, numpy) gives the same gradients.

The last test plants each mistake in the oracle's backward and requires a pin to catch it.
"""
import numpy as np
import pytest

import oracle
from tests._bruteforce import chunked_backward, reverse_scan, segment_reverse_fragments


def _unit_rows(rng, shape):
    x = rng.standard_normal(shape)
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _problem(seed, lengths, H, dk, dv, beta_zero=False):
    rng = np.random.default_rng(seed)
    T = int(sum(lengths))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    N = len(lengths)
    p = dict(q=rng.standard_normal((T, H, dk)), k=_unit_rows(rng, (T, H, dk)), v=rng.standard_normal((T, H, dv)),
             g=-np.abs(rng.standard_normal((T, H, dk))) * 0.2,
             beta=np.zeros((T, H)) if beta_zero else rng.uniform(0.05, 0.95, (T, H)),
             s0=rng.standard_normal((N, H, dk, dv)) * 0.3)
    do = rng.standard_normal((T, H, dv))
    dsT = rng.standard_normal((N, H, dk, dv))
    return p, cu, do, dsT, rng


def _loss(p, cu, do, dsT):
    r = oracle.recurrence(p["q"], p["k"], p["v"], p["g"], p["beta"], cu, s0=p["s0"])
    return float((r["o"] * do).sum() + (r["s_final"] * dsT).sum()), r


def _grads(p, cu, do, dsT, mut):
    return oracle.backward(p["q"], p["k"], p["v"], p["g"], p["beta"], cu, do, s0=p["s0"], ds_final=dsT,
                           mutation=mut)


GRAD_OF = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "s0": "ds0"}


def check_finite_differences(mut="none"):
    # lengths cross the oracle's 64-token checkpoints; dk != dv catches a transposed index
    p, cu, do, dsT, rng = _problem(11, [1, 63, 130], H=2, dk=6, dv=5)
    gr = _grads(p, cu, do, dsT, mut)
    eps = 1e-6
    for name, x in p.items():
        direction = rng.standard_normal(x.shape)
        plus, minus = dict(p), dict(p)
        plus[name] = x + eps * direction
        minus[name] = x - eps * direction
        fd = (_loss(plus, cu, do, dsT)[0] - _loss(minus, cu, do, dsT)[0]) / (2 * eps)
        an = float((gr[GRAD_OF[name]] * direction).sum())
        assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, fd, an)


def check_homogeneity(mut="none"):
    p, cu, do, dsT, _ = _problem(12, [5, 70], H=2, dk=8, dv=8)
    gr = _grads(p, cu, do, dsT, mut)
    L, r = _loss(p, cu, do, dsT)
    out_part = float((r["o"] * do).sum())
    assert abs(float((gr["dq"] * p["q"]).sum()) - out_part) <= 1e-11 * max(1.0, abs(out_part))
    lin = float((gr["dv"] * p["v"]).sum() + (gr["ds0"] * p["s0"]).sum())
    assert abs(lin - L) <= 1e-11 * max(1.0, abs(L))


def check_beta_zero_closed_form(mut="none"):
    p, cu, do, dsT, _ = _problem(13, [9, 4], H=2, dk=5, dv=7, beta_zero=True)
    gr = _grads(p, cu, do, dsT, mut)
    assert not gr["dk"].any() and not gr["dv"].any()
    for i in range(len(cu) - 1):
        for h in range(p["q"].shape[1]):
            t0, t1 = cu[i], cu[i + 1]
            alpha = np.exp(p["g"][t0:t1, h])            # [L, dk]
            P = np.cumprod(alpha, axis=0)               # prod_{u<=t} alpha_u
            S0 = p["s0"][i, h]
            Q, dO, K, V = p["q"][t0:t1, h], do[t0:t1, h], p["k"][t0:t1, h], p["v"][t0:t1, h]
            y = dO @ S0.T                               # (S_0 dO_t) per token, [L, dk]
            # dq_t = S_t dO_t = P_t * (S_0 dO_t)
            np.testing.assert_allclose(gr["dq"][t0:t1, h], P * y, rtol=1e-12, atol=1e-13)
            # dS_0 = sum_t Diag(P_t) q_t dO_t^T + Diag(P_T) dS_T
            ds0 = (P * Q).T @ dO + P[-1][:, None] * dsT[i, h]
            np.testing.assert_allclose(gr["ds0"][i, h], ds0, rtol=1e-12, atol=1e-12)
            # dg_u = sum_{t >= u} q_t * P_t * (S_0 dO_t) + P_T * rowsum(dS_T o S_0)
            per_t = Q * P * y
            dg = np.cumsum(per_t[::-1], axis=0)[::-1] + P[-1] * (dsT[i, h] * S0).sum(axis=1)
            np.testing.assert_allclose(gr["dg"][t0:t1, h], dg, rtol=1e-11, atol=1e-12)
            # dbeta_t = k_t^T D_t e_t, D_t = sum_{t' >= t} Diag(P_t'/P_t) q_t' dO_t'^T + Diag(P_T/P_t) dS_T,
            # e_t = v_t - (Diag(P_t) S_0)^T k_t
            for t in range(t1 - t0):
                D = sum((P[u] / P[t])[:, None] * np.outer(Q[u], dO[u]) for u in range(t, t1 - t0))
                D = D + (P[-1] / P[t])[:, None] * dsT[i, h]
                e = V[t] - (P[t][:, None] * S0).T @ K[t]
                assert abs(gr["dbeta"][t0 + t, h] - K[t] @ D @ e) <= 1e-11 * max(1.0, abs(K[t] @ D @ e))


def check_chunked_second_formulation(mut="none"):
    """The chunk-parallel backward algebra (numpy fp64, pair decays taken pairwise) equals the sequential one."""
    p, cu, do, dsT, _ = _problem(15, [150, 64, 3], H=2, dk=8, dv=6)
    p["g"] = p["g"] * 4  # steep gates: e^G spans ~1e-30 over a chunk
    gr = _grads(p, cu, do, dsT, mut)
    for i in range(len(cu) - 1):
        t0, t1 = cu[i], cu[i + 1]
        for h in range(2):
            cb = chunked_backward(*(p[n][t0:t1, h] for n in ("q", "k", "v", "g", "beta")), p["s0"][i, h],
                                  do[t0:t1, h], dsT[i, h])
            for n in ("dq", "dk", "dv", "dg", "dbeta"):
                ref = gr[n][t0:t1, h]
                assert np.abs(cb[n] - ref).max() <= 1e-11 * max(1.0, np.abs(ref).max()), (n, i, h)
            assert np.abs(cb["ds0"] - gr["ds0"][i, h]).max() <= 1e-11 * max(1.0, np.abs(gr["ds0"][i, h]).max())


PINS = [check_finite_differences, check_homogeneity, check_beta_zero_closed_form, check_chunked_second_formulation]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_backward_pin(pin):
    pin()


def test_backward_empty_sequences_pass_the_state_gradient_through():
    """A zero-length sequence has S_T = S_0, so its dS_0 is dS_T unchanged (one-token sequences are in the
    finite-difference pin)."""
    p, cu, do, dsT, _ = _problem(14, [0, 1, 0], H=1, dk=4, dv=3)
    gr = _grads(p, cu, do, dsT, "none")
    np.testing.assert_array_equal(gr["ds0"][0], dsT[0])
    np.testing.assert_array_equal(gr["ds0"][2], dsT[2])


@pytest.mark.parametrize("mut", [m for m in oracle.BACKWARD_MUTATIONS if m != "none"])
def test_planted_backward_mistakes_are_caught(mut):
    caught = []
    for pin in PINS:
        try:
            pin(mut)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {mut}"


def test_segmented_reverse_carry_matches_suffix_backwards():
    """The backward's state-gradient carry splits into segments like the forward's state: per segment a
    fragment (N, b~) with dS_in = N dS_out + b~, composed by a scan from dS_T (tests/_bruteforce.py).  At
    every segment boundary t_p the scan's gradient must equal dL/dS_{t_p} from the oracle's own backward
    over the suffix [t_p, T) started from the forward state at t_p (outputs before t_p do not depend on
    S_{t_p}), and at t = 0 the oracle's dS_0 over the whole sequence; then each segment's reverse pass from
    its exact exit gradient and forward entry state reproduces the whole backward's gradients."""
    p, cu, do, dsT, _ = _problem(16, [300], H=2, dk=8, dv=6)
    T, C, seg = 300, 64, 2
    names = ("q", "k", "v", "g", "beta")
    gr = _grads(p, cu, do, dsT, "none")
    bounds = list(range(0, T, C * seg))  # segment starts: 0, 128, 256
    for h in range(2):
        frags = segment_reverse_fragments(*(p[n][:, h] for n in names), do[:, h], C=C, seg_chunks=seg)
        grads = reverse_scan(frags, dsT[0, h])  # exit gradient of each segment, then dL/dS_0
        assert len(frags) == len(bounds)
        np.testing.assert_allclose(grads[-1], gr["ds0"][0, h], rtol=1e-10, atol=1e-12)
        for sp, t_p in enumerate(bounds[1:]):  # the exit gradient of segment sp is dL/dS_{t_p}
            head = oracle.recurrence(*(p[n][:t_p] for n in names), [0, t_p], s0=p["s0"][:1])
            suffix = oracle.backward(*(p[n][t_p:] for n in names), [0, T - t_p], do[t_p:],
                                     s0=head["s_final"], ds_final=dsT[:1])
            np.testing.assert_allclose(grads[sp], suffix["ds0"][0, h], rtol=1e-10, atol=1e-12)
        # each segment's reverse pass from its exact exit gradient and forward entry state
        for sp, t0 in enumerate(bounds):
            t1 = min(t0 + C * seg, T)
            entry = p["s0"][0, h] if t0 == 0 else oracle.recurrence(
                *(p[n][:t0, h:h + 1] for n in names), [0, t0], s0=p["s0"][:1, h:h + 1])["s_final"][0, 0]
            cb = chunked_backward(*(p[n][t0:t1, h] for n in names), entry, do[t0:t1, h], grads[sp])
            for n in ("dq", "dk", "dv", "dg", "dbeta"):
                ref = gr[n][t0:t1, h]
                assert np.abs(cb[n] - ref).max() <= 1e-10 * max(1.0, np.abs(ref).max()), (n, sp, h)
