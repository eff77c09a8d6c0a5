"""Helpers for the GPU parity tests: move seeded inputs to the device, run the library through its binding,
run the oracle on the same bytes, and measure the error the way the tolerances are stated
(max |difference| over all compared values divided by the rms of the oracle's values)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth


def dev(x: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x))
    if x.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.cuda()


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return synth.bf16_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def rel_err(got, ref) -> float:
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    return float(np.max(np.abs(got - ref)) / rms) if ref.size else 0.0


def status(t: torch.Tensor):
    s = t.cpu().numpy()
    return int(s[0]), int(np.uint32(s[1]))


class PrefillRun:
    """Device copies of a synth.Prefill problem plus the outputs of one library call."""

    def __init__(self, prob: synth.Prefill, out_dtype=torch.float32):
        self.prob = prob
        self.q, self.k, self.v = dev(prob.q), dev(prob.k), dev(prob.v)
        self.g, self.beta = dev(prob.g), dev(prob.beta)
        self.cu = dev(prob.cu_seqlens.astype(np.int32))
        self.pool = dev(prob.pool)
        self.slots = dev(prob.slot_ids.astype(np.int32))
        self.out = torch.zeros(prob.T, prob.H, prob.dv, dtype=out_dtype, device="cuda")
        self.extra = self.extra_slots = None
        if prob.extra_pool is not None:
            self.extra = dev(prob.extra_pool)
            self.extra_slots = dev(prob.extra_slot_ids.astype(np.int32))
        self.status = torch.zeros(2, dtype=torch.int32, device="cuda")
        self.max_seqlen = int(max(prob.lengths.max(), 0)) if prob.N else 0

    def common(self):
        return dict(init_zero=self.prob.init_zero, extra_pool=self.extra, extra_slot_ids=self.extra_slots,
                    snapshot_every_chunks=self.prob.snapshot_every_chunks if self.extra is not None else 0,
                    dev_status=self.status)

    def args(self):
        return (self.q, self.k, self.v, self.g, self.beta, self.cu, self.max_seqlen, self.pool, self.slots, self.out)

    def varlen_workspace(self, kda):
        n = kda.kda_prefill_workspace_size(*self.args(),
                                           **{k: v for k, v in self.common().items() if k != "dev_status"})
        return torch.empty(n, dtype=torch.uint8, device="cuda") if n else None

    def run_varlen(self, kda):
        kda.kda_prefill_varlen(*self.args(), workspace=self.varlen_workspace(kda), **self.common())
        torch.cuda.synchronize()
        return self

    def workspace_for(self, kda, segment_len):
        n = kda.kda_segmented_workspace_size(*self.args(), segment_len,
                                             **{k: v for k, v in self.common().items() if k != "dev_status"})
        return torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")

    def run_segmented(self, kda, segment_len):
        ws = self.workspace_for(kda, segment_len)
        kda.kda_prefill_segmented(*self.args(), segment_len, ws, **self.common())
        torch.cuda.synchronize()
        return self


def oracle_prefill(prob: synth.Prefill, want_o=True, sample_t=None, threads=0):
    s0 = None if prob.init_zero else prob.pool[prob.slot_ids].astype(np.float64)
    every = prob.snapshot_every_chunks * 64 if (prob.extra_pool is not None and prob.snapshot_every_chunks) else 0
    return oracle.recurrence(prob.q, prob.k, prob.v, prob.g, prob.beta, prob.cu_seqlens, s0=s0, want_o=want_o,
                             sample_t=sample_t, snap_every=every, threads=threads)


def expected_extra_pool(prob: synth.Prefill, ref) -> np.ndarray:
    """Contents of the ping-pong extra pool after the prefill: snapshot m of sequence i sits in entry
    (m - 1) & 1 of its pair; later snapshots overwrite earlier ones in the same entry."""
    extra = prob.extra_pool.astype(np.float64).copy()
    for i, snaps in enumerate(ref.get("snaps", [])):
        for m in range(1, len(snaps) + 1):
            extra[prob.extra_slot_ids[i, (m - 1) & 1]] = snaps[m - 1]
    return extra


def prefix_problem(prob, i: int, ntok: int):
    """Sequence i of `prob` cut to its first ntok tokens, alone in the batch, from the same initial state
    (same pool and slot), with no snapshots."""
    a = int(prob.cu_seqlens[i])
    sl = lambda x: np.ascontiguousarray(x[a:a + ntok])
    return synth.Prefill("prefix", prob.seed, prob.H, prob.dk, prob.dv, prob.in_dtype, sl(prob.q), sl(prob.k),
                         sl(prob.v), sl(prob.g), sl(prob.beta), np.array([0, ntok], np.int32), prob.pool,
                         prob.slot_ids[i:i + 1].copy(), init_zero=prob.init_zero)
