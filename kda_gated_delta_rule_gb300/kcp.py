"""KCP across GPUs: one long sequence split into contiguous shards, one shard per rank.

Source: "Kimi K3 training and serving infra" (marsggbo blog), section 4.2 "KCP: pass fixed-size transition
information".  Each rank reduces its shard to a fixed-size fragment (the state S~ the shard produces from a
zero input state, and its cumulative transition M), the ranks exchange the fragments with one all-gather
(2 x 64 KB per head at d = 128, whatever the shard length), every rank scans them to its exact entry state
(entry_0 = S_0, entry_{r+1} = M_r entry_r + S~_r), and computes its outputs.  The compute steps are the
library's kernels (kda_kcp_fragments, kda_kcp_scan, kda_kcp_outputs); the exchange is torch.distributed's
all-gather over the process group (NCCL between GPUs).  Every rank computes the same scan on the same
gathered bytes, so the entry states agree bit for bit across ranks.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist

from . import kda_kcp_fragments, kda_kcp_outputs, kda_kcp_scan, kda_prefill_records, kda_segmented_workspace_size


class LibraryOps:
    """The per-rank compute of KCP on this rank's GPU.  q, k, v, g, beta are the shard's token-major inputs
    [L, H, d] (one sequence of L > 0 tokens)."""

    def __init__(self, q, k, v, g, beta, out, final_state):
        self.inp = (q, k, v, g, beta)
        L, H, d = q.shape
        dev = q.device
        self.cu = torch.tensor([0, L], dtype=torch.int32, device=dev)
        self.L = L
        self.seg = ((L + 63) // 64) * 64              # one segment: the whole shard
        self.pool = final_state.view(1, H, d, d)      # the shard's final state is written here
        self.slots = torch.zeros(1, dtype=torch.int32, device=dev)
        self.out = out
        n = kda_segmented_workspace_size(*self.inp, self.cu, L, self.pool, self.slots, out, self.seg)
        self.ws = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
        self.H, self.d = H, d

    def _args(self):
        return (*self.inp, self.cu, self.L, self.pool, self.slots, self.out)

    def fragments(self):
        kda_prefill_records(*self._args(), workspace=self.ws)
        frag = torch.empty(1, 1, self.H, self.d, 2 * self.d, device=self.out.device)
        kda_kcp_fragments(*self._args(), self.seg, self.ws, frag)
        return frag[0, 0]

    def scan(self, frags, s0):
        entries = torch.empty(frags.shape[0], self.H, self.d, self.d, device=frags.device)
        kda_kcp_scan(frags, s0, entries)
        return entries

    def outputs(self, entry):
        kda_kcp_outputs(*self._args(), self.seg, self.ws, entry.contiguous().view(1, 1, self.H, self.d, self.d))


def kcp_prefill(ops, s0, group=None):
    """Runs this rank's part of a sequence-sharded prefill and returns the entry states of all ranks
    [W, H, d, d].  `ops` carries the shard (LibraryOps on a GPU); s0 [H, d, d] is the sequence's initial
    state, the same on every rank (or None for zero)."""
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    frag = ops.fragments().contiguous()
    parts = [torch.empty_like(frag) for _ in range(world)]
    dist.all_gather(parts, frag, group=group)
    frags = torch.stack(parts)  # rank order = token order
    entries = ops.scan(frags, s0)
    ops.outputs(entries[rank])
    return entries


def shard_bounds(T: int, world: int) -> np.ndarray:
    """Token offsets of `world` contiguous shards of a T-token sequence, as equal as possible (T >= world)."""
    return np.array([(T * r) // world for r in range(world + 1)], np.int64)
