"""Operand precision of the chunked prefill's tensor-core products (CPU; no GPU needed).

Per chunk of 64 tokens with entry state S the chain computes U = U~ - W S, O = Qh S + P U and
S' = Diag(gamma_C) S + Kh^T U (the chunk algebra of the recurrence in the "Kimi K3: Architecture and SGLang
Day-0 Support" KDA math box, derived by induction over a chunk's tokens), with W, Qh, P and Kh read from the
chunk records and S and U split in tensor memory.  Every product takes both operands as bf16 hi + lo
(hi*hi + lo*hi + hi*lo) and U~ stays fp32.  This test fixes, on the 8K workload's distributions (two heads
of it, 128 chunks each), what that costs against the 2e-3 x rms bound, measured against the fp64 oracle,
and what dropping the lo half of any one operand would cost: for every operand but W the error passes the
bound, and W alone takes more than a quarter of it (while saving 16 of a chunk record's 144 KB), so a
smaller record cannot come from a narrower operand format.
"""
import numpy as np
import pytest

import oracle
import synth
from tests._precision import f32, product

BOUND = 2e-3
T, H, C = 8192, 2, 64


@pytest.fixture(scope="module")
def chunks():
    prob = synth.prefill_8k(T=T, H=H)
    f = lambda x: synth.bf16_to_f32(x).astype(np.float64) if x.dtype == np.uint16 else x.astype(np.float64)
    q, k, v = f(prob.q), f(prob.k), f(prob.v)
    g, beta = prob.g.astype(np.float64), prob.beta.astype(np.float64)
    s0 = prob.pool[prob.slot_ids].astype(np.float64)
    ref = oracle.recurrence(prob.q, prob.k, prob.v, prob.g, prob.beta, prob.cu_seqlens, s0=s0)
    strict = np.tril(np.ones((C, C)), -1)[:, :, None] > 0
    incl = np.tril(np.ones((C, C)))[:, :, None] > 0
    recs = []
    for h in range(H):
        rh = []
        for c0 in range(0, T, C):
            sl = slice(c0, c0 + C)
            qc, kc, vc, bc = q[sl, h], k[sl, h], v[sl, h], beta[sl, h]
            G = np.cumsum(g[sl, h], axis=0)
            E = np.exp(G[:, None, :] - G[None, :, :])  # pair decays e^(G_t - G_s), used for s <= t
            A = np.einsum("tj,sj,tsj->ts", kc, kc, np.where(strict, E, 0.0)) * bc[:, None]
            P = np.einsum("tj,sj,tsj->ts", qc, kc, np.where(incl, E, 0.0))
            Tinv = np.linalg.inv(np.eye(C) + A)
            rh.append(dict(W=Tinv @ (bc[:, None] * kc * np.exp(G)), Ut=f32(Tinv @ (bc[:, None] * vc)),
                           Qh=qc * np.exp(G), P=P, KhT=(kc * np.exp(G[-1] - G)).T, gC=np.exp(G[-1])))
        recs.append(rh)
    return s0[0], recs, ref


def _chain(chunks, **single):
    """Runs the chain with every operand split, except those named in `single` (single bf16)."""
    s0, recs, ref = chunks
    fmt = lambda name: "bf16" if single.get(name) else "split"
    O = np.zeros_like(ref["o"])
    SF = np.zeros((H,) + s0.shape[1:])
    for h in range(H):
        S = s0[h].copy()
        for ci, r in enumerate(recs[h]):
            U = f32(r["Ut"] - product(r["W"], S, fmt("W"), fmt("S")))
            O[ci * C:(ci + 1) * C, h] = product(r["Qh"], S, fmt("Qh"), fmt("S")) + product(r["P"], U, fmt("P"),
                                                                                          fmt("U"))
            S = f32(r["gC"][:, None] * S + product(r["KhT"], U, fmt("Kh"), fmt("U")))
        SF[h] = S
    e_o = np.max(np.abs(O - ref["o"])) / np.sqrt(np.mean(ref["o"] ** 2))
    e_s = np.max(np.abs(SF - ref["s_final"][0])) / np.sqrt(np.mean(ref["s_final"] ** 2))
    return float(e_o), float(e_s)


def test_split_operands_stay_well_inside_the_bound(chunks):
    e_o, e_s = _chain(chunks)
    assert e_o <= BOUND / 10 and e_s <= BOUND / 10, (e_o, e_s)


@pytest.mark.parametrize("operand", ["S", "Qh", "P", "U", "Kh"])
def test_a_single_bf16_operand_breaks_the_bound(chunks, operand):
    e_o, e_s = _chain(chunks, **{operand: True})
    assert max(e_o, e_s) > BOUND, (operand, e_o, e_s)


def test_a_single_bf16_w_takes_over_a_quarter_of_the_bound(chunks):
    e_o, e_s = _chain(chunks, W=True)
    assert max(e_o, e_s) > BOUND / 4, (e_o, e_s)
