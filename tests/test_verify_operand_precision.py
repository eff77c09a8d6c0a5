"""Operand precision of the verify window's state product (CPU; no GPU needed).

The tensor-core verify computes each window as O = Qh S0 + Oh, with Qh = Q o e^G - R (K o e^G),
Oh = R V and R = P (I + A)^-1 diag(beta) (the chunk algebra of the recurrence in the "Kimi K3:
Architecture and SGLang Day-0 Support" KDA math box, applied to one window from the committed state).
The state product runs on the tensor cores, so its operands take a tensor-core format.  This test fixes,
on windows drawn like the decode + verify workload's (bf16 inputs, W = 8, H = 12, d = 128), what each
operand format costs against the 2e-3 x rms(o) bound, measured against the fp64 oracle:

* single bf16 operands use up more than half of the bound on their own, so the kernel splits both
  operands into bf16 hi + lo and forms hi*hi + lo*hi + hi*lo (error ~1e-5);
* tf32 operands (10 stored mantissa bits), truncated or rounded, stay within half of the bound: a
  single-pass tf32 product is an admissible alternative for the state side.
"""
import numpy as np

import oracle
import synth
from tests._precision import bf16 as bf16_rne, tf32_round, tf32_trunc

BOUND = 2e-3


def _window_terms(p):
    """Qh and Oh of every (request, head) window, in fp64 from the chunk algebra."""
    B, W, H, d = p.B, p.W, p.H, p.dk
    f = lambda x: synth.bf16_to_f32(x).astype(np.float64) if x.dtype == np.uint16 else x.astype(np.float64)
    Q, K, V = f(p.wq), f(p.wk), f(p.wv)
    G = np.cumsum(p.wg.astype(np.float64), axis=1)  # in-window cumulative log-decay
    beta = p.wbeta.astype(np.float64)
    Qh, Oh = np.zeros((B, W, H, d)), np.zeros((B, W, H, d))
    for h in range(H):
        q, k, v, g, bt = Q[:, :, h], K[:, :, h], V[:, :, h], G[:, :, h], beta[:, :, h]
        kp, km = k * np.exp(g), k * np.exp(-g)
        P = np.tril(np.matmul(q * np.exp(g), km.transpose(0, 2, 1)))          # u <= t
        A = np.tril(np.matmul(kp, km.transpose(0, 2, 1)), -1) * bt[:, :, None]  # u < t
        R = np.matmul(P, np.linalg.inv(np.eye(W)[None] + A)) * bt[:, None, :]
        Qh[:, :, h] = q * np.exp(g) - np.matmul(R, kp)
        Oh[:, :, h] = np.matmul(R, v)
    return Qh, Oh


def test_state_product_operand_formats():
    p = synth.decode_verify(seed=4, B=32, W=8, H=12, d=128, num_slots=32)
    B, W, H, d = p.B, p.W, p.H, p.dk
    flat = lambda x: np.ascontiguousarray(x.reshape((B * W,) + x.shape[2:]))
    ref = oracle.recurrence(flat(p.wq), flat(p.wk), flat(p.wv), flat(p.wg), flat(p.wbeta),
                            np.arange(0, B * W + 1, W), s0=p.pool[p.slot_ids], want_final=False)["o"]
    ref = ref.reshape(B, W, H, d)
    rms = np.sqrt(np.mean(ref ** 2))
    S0 = p.pool[p.slot_ids].astype(np.float64)
    Qh, Oh = _window_terms(p)

    def prod(qh, s0):
        return np.matmul(qh.transpose(0, 2, 1, 3), s0).transpose(0, 2, 1, 3)

    err = lambda o: float(np.max(np.abs(o - ref)) / rms)
    assert err(prod(Qh, S0) + Oh) <= 1e-12  # the window algebra itself is exact
    sh, qh = bf16_rne(S0), bf16_rne(Qh)
    split = prod(qh, sh) + prod(bf16_rne(Qh - qh), sh) + prod(qh, bf16_rne(S0 - sh)) + Oh
    assert err(split) <= 5e-5
    assert err(prod(bf16_rne(Qh), bf16_rne(S0)) + Oh) > BOUND / 2
    assert err(prod(tf32_trunc(Qh), tf32_trunc(S0)) + Oh) <= BOUND / 2
    assert err(prod(tf32_round(Qh), tf32_round(S0)) + Oh) <= BOUND / 4
