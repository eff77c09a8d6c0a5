"""Fused decode front/back-end (short convolution + KDA step + gated output norm) against the fp64 oracle.

Several consecutive tokens per request, carrying both the KDA state and the convolution inputs through the
pool.  fp32 outputs and states within 2e-3 of the oracle's rms (the forward's bar); a bf16 output is the
round-to-nearest-even of the fp32 one, bit for bit (the rounding alone exceeds 2e-3 of the rms); the
carried convolution inputs are copies of the token inputs, so they must match bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests._gpu import dev, host, rel_err, status

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.mark.parametrize("B,H,S,steps", [(6, 3, 10, 4), (48, 8, 64, 2)], ids=["B6H3", "B48H8"])
@pytest.mark.parametrize("dtype", [synth.BF16, synth.F32], ids=["bf16", "f32"])
def test_fused_decode_steps_match_oracle(cuda, dtype, B, H, S, steps):
    """B48H8: 384 (request, head) units, more than the two persistent CTAs per SM take in one round."""
    d = 128
    p = synth.fused_decode_inputs(71, B, H, d, S, steps, dtype)
    pool, cstate = dev(p["pool"]), dev(p["conv_state"])
    slots, cw, nw = dev(p["slot_ids"]), dev(p["conv_w"]), dev(p["norm_w"])
    ref_pool = p["pool"].astype(np.float64)
    ref_cs = p["conv_state"].astype(np.float64)
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    for t in range(steps):
        xs = [dev(p[n][t]) for n in ("xq", "xk", "xv", "a", "b", "z")]
        out16 = torch.empty(B, H, d, dtype=torch.bfloat16, device="cuda")
        cuda.kda_fused_decode(*xs, pool.clone(), slots, cstate.clone(), cw, nw, out16, norm_eps=1e-5)
        out = torch.empty(B, H, d, dtype=torch.float32, device="cuda")
        cuda.kda_fused_decode(*xs, pool, slots, cstate, cw, nw, out, norm_eps=1e-5, dev_status=st)
        y, states, new_cs = oracle.fused_decode(ref_pool, ref_cs, p["slot_ids"], *(p[n][t] for n in
                                                ("xq", "xk", "xv", "a", "b", "z")), p["conv_w"], p["norm_w"], 1e-5)
        ref_pool[p["slot_ids"]] = states
        ref_cs[p["slot_ids"]] = new_cs
        torch.cuda.synchronize()
        assert rel_err(host(out), y) <= TOL, t
        assert torch.equal(out16, out.to(torch.bfloat16)), t
    assert status(st) == (0, steps * B * H)
    assert rel_err(host(pool)[p["slot_ids"]], ref_pool[p["slot_ids"]]) <= TOL
    np.testing.assert_array_equal(host(cstate), ref_cs)  # untouched slots included


def test_fused_decode_bad_slot_is_flagged_and_skipped(cuda):
    B, H, d, S = 2, 1, 128, 4
    p = synth.fused_decode_inputs(72, B, H, d, S)
    slots = p["slot_ids"].copy()
    slots[1] = S + 5
    pool, cstate = dev(p["pool"]), dev(p["conv_state"])
    out = torch.zeros(B, H, d, device="cuda")
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    cuda.kda_fused_decode(*(dev(p[n][0]) for n in ("xq", "xk", "xv", "a", "b", "z")), pool, dev(slots), cstate,
                          dev(p["conv_w"]), dev(p["norm_w"]), out, dev_status=st)
    torch.cuda.synchronize()
    assert status(st) == (cuda.KDA_DEV_SLOT_OOB, H)
    assert not out[1].any()
    untouched = [s for s in range(S) if s != slots[0]]
    np.testing.assert_array_equal(host(pool)[untouched], p["pool"][untouched])
    np.testing.assert_array_equal(host(cstate)[untouched], p["conv_state"][untouched])


def test_fused_decode_skips_bad_units_mid_stream(cuda):
    """512 (request, head) units, several per persistent CTA, with bad slot ids scattered through the batch:
    flagged and left alone; every other unit gets the bits of a call on the good requests only."""
    B, H, d, S = 64, 8, 128, 80
    p = synth.fused_decode_inputs(73, B, H, d, S)
    bad_rows = np.array([0, 31, 63])
    good = np.setdiff1d(np.arange(B), bad_rows)
    slots = p["slot_ids"].copy()
    slots[bad_rows] = [S, -1, S + 100]
    xs = [dev(p[n][0]) for n in ("xq", "xk", "xv", "a", "b", "z")]
    cw, nw = dev(p["conv_w"]), dev(p["norm_w"])
    pool, cstate = dev(p["pool"]), dev(p["conv_state"])
    out = torch.zeros(B, H, d, device="cuda")
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    cuda.kda_fused_decode(*xs, pool, dev(slots), cstate, cw, nw, out, dev_status=st)
    gi = torch.from_numpy(good).cuda()
    pool_g, cstate_g = dev(p["pool"]), dev(p["conv_state"])
    out_g = torch.zeros(len(good), H, d, device="cuda")
    cuda.kda_fused_decode(*(x[gi].contiguous() for x in xs), pool_g, dev(p["slot_ids"][good]), cstate_g, cw, nw, out_g)
    torch.cuda.synchronize()
    assert status(st) == (cuda.KDA_DEV_SLOT_OOB, len(good) * H)
    assert torch.equal(out[gi], out_g) and not out[torch.from_numpy(bad_rows).cuda()].any()
    assert torch.equal(pool, pool_g) and torch.equal(cstate, cstate_g)
