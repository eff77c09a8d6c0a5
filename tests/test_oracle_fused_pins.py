"""Pins for the oracle's fused decode front/back-end (short convolution, normalisations, gates, output norm).

* The stepwise short convolution with its carried inputs equals the full causal convolution of the whole
  sequence computed by numpy (np.convolve), followed by SiLU; the carried state is the last W-1 inputs.
* The composed path reproduces the read-back identity of the KDA math box ("Kimi K3: Architecture and
  SGLang Day-0 Support"): for a unit key, S_t^T k_t = (1 - beta) r_old + beta v_t.  With x_q = x_k and equal
  convolution taps the normalised query equals the normalised key, so beta -> 1 makes the read-out exactly
  v_t whatever the state, and the output is v_t scaled to unit rms, times the norm weight and the gate.
* Gate limits: the log-decay stays inside (g_min, 0); beta -> 0 and g -> 0 leave the state unchanged.
* Output norm and gates (the pages fix no formula for them, so their properties are pinned, not their
  expressions): unit rms after dividing out the weight and the gate, invariance to the read-out's scale
  (and oddness in it) at eps = 0, eps shrinking small read-outs most; the output gate's open, midpoint and
  closed limits; the weight scaling its channel; the decay gate's floor e^{-5}, midpoint e^{-2.5} and
  open limit seen through the new state, per key channel.
"""
import numpy as np

import oracle


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def test_stepwise_conv_equals_full_causal_convolution():
    rng = np.random.default_rng(3)
    T, C, W = 23, 5, oracle.CONV_WIDTH
    x = rng.standard_normal((T, C))
    w = rng.standard_normal((C, W))  # asymmetric taps: a reversed window would not match
    state = np.zeros((C, W - 1))
    for t in range(T):
        y, state = oracle.short_conv_step(x[t], state, w)
        for c in range(C):
            # causal convolution: sum_tau w[c, W-1-tau] x[t - tau, c]
            full = np.convolve(x[:t + 1, c], w[c, ::-1])[t]
            assert abs(y[c] - full * _sigmoid(full)) <= 1e-12 * max(1.0, abs(full))
        np.testing.assert_array_equal(state, x[max(0, t - W + 2):t + 1].T if t >= W - 2 else
                                      np.concatenate([np.zeros((C, W - 2 - t)), x[:t + 1].T], axis=1))


def _problem(rng, B=3, H=2, d=8, S=6):
    slots = np.array([4, 0, 2])[:B]
    return dict(pool=rng.standard_normal((S, H, d, d)) * 0.3,
                conv_state=rng.standard_normal((S, H, 3, oracle.CONV_WIDTH - 1, d)),
                slot_ids=slots, xq=rng.standard_normal((B, H, d)), xk=rng.standard_normal((B, H, d)),
                xv=rng.standard_normal((B, H, d)), a=rng.standard_normal((B, H, d)), b=rng.standard_normal((B, H)),
                z=rng.standard_normal((B, H, d)), conv_w=rng.standard_normal((3, 2, d, oracle.CONV_WIDTH)),
                norm_w=rng.uniform(0.5, 1.5, d), eps=1e-5)


def test_readback_identity_through_the_fused_path():
    rng = np.random.default_rng(4)
    p = _problem(rng)
    p["xk"] = p["xq"].copy()
    p["conv_w"][1] = p["conv_w"][0]
    p["conv_state"][:, :, 1] = p["conv_state"][:, :, 0]   # same carried inputs for q and k
    p["b"] = np.full_like(p["b"], 40.0)                      # beta = 1 - 4e-18
    y, _, new_cs = oracle.fused_decode(**p)
    # v_t = SiLU(conv(x_v)) from the carried v inputs
    cs = p["conv_state"][p["slot_ids"]]
    window = np.concatenate([np.moveaxis(cs[:, :, 2], -2, -1), p["xv"][..., None]], axis=-1)
    yv = (window * p["conv_w"][2]).sum(-1)
    v = yv * _sigmoid(yv)
    expect = v / np.sqrt((v * v).mean(-1, keepdims=True) + p["eps"]) * p["norm_w"] * _sigmoid(p["z"])
    np.testing.assert_allclose(y, expect, rtol=0, atol=1e-5)  # |k| = 1 up to the 1e-6 in the normalisation
    # the carried inputs advance by one: the new window is (x_{t-2}, x_{t-1}, x_t)
    np.testing.assert_array_equal(new_cs[:, :, 2, :-1], cs[:, :, 2, 1:])
    np.testing.assert_array_equal(new_cs[:, :, 2, -1], p["xv"])


def test_gates_inside_bounds_and_a_closed_gate_keeps_the_state():
    rng = np.random.default_rng(5)
    p = _problem(rng)
    a = np.linspace(-30, 30, 101)
    g = oracle.G_MIN * _sigmoid(a)
    assert np.all(g > oracle.G_MIN) and np.all(g < 0)
    p["a"] = np.full_like(p["a"], -60.0)   # g ~ -4e-26: alpha = 1
    p["b"] = np.full_like(p["b"], -60.0)   # beta ~ 9e-27
    _, states, _ = oracle.fused_decode(**p)
    np.testing.assert_allclose(states, p["pool"][p["slot_ids"]], rtol=0, atol=1e-20)


# The pages name the fused Conv + KDA + output-norm decode kernel and say the log-decay is kept above
# g_min = -5 by a scaled sigmoid and that the output is gated, but they print no formula for the norm or
# the gates.  The pins below therefore fix properties of the reading taken (an RMS normalisation of the
# read-out, a per-channel weight, a sigmoid output gate, a sigmoid-scaled log-decay with floor g_min),
# checked through the whole composed path without re-evaluating the oracle's own expressions.

def _quiet(p):
    """Closed write gate (beta ~ 1e-26): the read-out is S~^T q, linear in the carried state."""
    p = dict(p)
    p["b"] = np.full_like(p["b"], -60.0)
    return p


def test_output_norm_is_scale_free_with_unit_rms():
    rng = np.random.default_rng(6)
    p = _quiet(_problem(rng))
    p["eps"] = 0.0
    y, _, _ = oracle.fused_decode(**p)
    gate = p["norm_w"] * _sigmoid(p["z"])
    # unit rms once the weight and the gate are divided out
    np.testing.assert_allclose(np.sqrt(((y / gate) ** 2).mean(-1)), 1.0, rtol=1e-12)
    # scale-free and odd in the read-out: scaling the carried state scales o (beta ~ 0), y does not move
    for c in (1e-3, 7.5, -2.0):
        pc = dict(p)
        pc["pool"] = p["pool"] * c
        yc, _, _ = oracle.fused_decode(**pc)
        np.testing.assert_allclose(yc, np.sign(c) * y, rtol=1e-10, atol=1e-12)
    # eps > 0 shrinks the output towards zero, more for a small read-out than for a large one
    pe = dict(p)
    pe["eps"] = 1e-2
    small = dict(pe)
    small["pool"] = p["pool"] * 1e-3
    ye, _, _ = oracle.fused_decode(**pe)
    ys, _, _ = oracle.fused_decode(**small)
    assert np.all(np.abs(ye) <= np.abs(y) + 1e-15) and np.all(np.abs(ys) <= np.abs(ye) + 1e-15)
    assert np.max(np.abs(ys)) < 0.5 * np.max(np.abs(ye))


def test_output_weight_and_gate_limits():
    rng = np.random.default_rng(7)
    p = _problem(rng)
    p["z"] = np.full_like(p["z"], 60.0)        # open gate: sigmoid = 1 - 9e-27
    y_open, _, _ = oracle.fused_decode(**p)
    p2 = dict(p)
    p2["z"] = np.zeros_like(p["z"])            # the midpoint of a sigmoid gate halves the output
    y_half, _, _ = oracle.fused_decode(**p2)
    np.testing.assert_allclose(y_half, 0.5 * y_open, rtol=1e-12, atol=1e-15)
    p3 = dict(p)
    p3["z"] = np.full_like(p["z"], -60.0)      # a closed gate silences the output
    y_shut, _, _ = oracle.fused_decode(**p3)
    assert np.max(np.abs(y_shut)) < 1e-20
    p4 = dict(p)
    p4["norm_w"] = 2.0 * p["norm_w"]           # the per-channel weight scales its channel
    y_w, _, _ = oracle.fused_decode(**p4)
    np.testing.assert_allclose(y_w, 2.0 * y_open, rtol=1e-12, atol=1e-15)


def test_decay_gate_floor_and_midpoint_through_the_state():
    """With the write gate closed, the new state is Diag(alpha) S: a -> +inf reaches the floor alpha =
    e^{g_min} = e^{-5}, a = 0 gives the sigmoid's midpoint e^{-2.5}, a -> -inf keeps the state."""
    rng = np.random.default_rng(8)
    p = _quiet(_problem(rng))
    s0 = p["pool"][p["slot_ids"]]
    for a_val, alpha in ((60.0, np.exp(-5.0)), (0.0, np.exp(-2.5)), (-60.0, 1.0)):
        pa = dict(p)
        pa["a"] = np.full_like(p["a"], a_val)
        _, states, _ = oracle.fused_decode(**pa)
        np.testing.assert_allclose(states, alpha * s0, rtol=1e-12, atol=1e-20)
    # a per-channel decay scales the state's rows (key channels), not its columns
    pa = dict(p)
    pa["a"] = np.where(np.arange(p["a"].shape[-1]) % 2 == 0, 60.0, -60.0) * np.ones_like(p["a"])
    _, states, _ = oracle.fused_decode(**pa)
    row_scale = np.where(np.arange(s0.shape[-2]) % 2 == 0, np.exp(-5.0), 1.0)[:, None]
    np.testing.assert_allclose(states, row_scale * s0, rtol=1e-12, atol=1e-20)
