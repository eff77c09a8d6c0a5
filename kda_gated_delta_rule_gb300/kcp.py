"""KCP across GPUs: one long sequence split into contiguous shards, one shard per rank.

Source: "Kimi K3 training and serving infra" (marsggbo blog), section 4.2 "KCP: pass fixed-size transition
information".  Each rank cuts its shard into P segments of a common length and reduces every segment to a
fixed-size fragment (the state S~ the segment produces from a zero input state, and its cumulative
transition M), so that no rank walks its whole shard as one dependent chain.  The ranks exchange the
fragments with one all-gather (P x 2 x 64 KB per head at d = 128, whatever the shard length); every rank
scans all W x P fragments in token order to the exact entry state of every segment (entry_0 = S_0,
entry_{s+1} = M_s entry_s + S~_s) and computes its outputs from its own segments' entry states.  The compute
steps are the library's kernels (kda_kcp_fragments, kda_kcp_scan, kda_kcp_outputs); the exchange is
torch.distributed's all-gather over the process group (NCCL between GPUs).  Every rank computes the same
scan on the same gathered bytes, so the entry states agree bit for bit across ranks.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist

from . import kda_kcp_fragments, kda_kcp_outputs, kda_kcp_scan, kda_prefill_records, kda_segmented_workspace_size


def kcp_segment_len(T: int, world: int, segments_per_rank: int) -> int:
    """A segment length (multiple of 64) that cuts every rank's shard of a T-token sequence into the same
    number of segments, about `segments_per_rank` of them (the all-gather needs equal counts; the shards
    of shard_bounds differ by at most one token)."""
    b = shard_bounds(T, world)
    sizes = np.diff(b)
    lo, hi = int(sizes.min()), int(sizes.max())
    seg = max(64, -(-hi // (64 * max(1, segments_per_rank))) * 64)
    while -(-lo // seg) != -(-hi // seg):
        seg += 64
    return seg


class LibraryOps:
    """The per-rank compute of KCP on this rank's GPU.  q, k, v, g, beta are the shard's token-major inputs
    [L, H, d] (one sequence of L > 0 tokens); segment_len (a multiple of 64, the same on every rank, see
    kcp_segment_len) cuts the shard into P segments (None: one segment, the whole shard)."""

    def __init__(self, q, k, v, g, beta, out, final_state, segment_len=None):
        self.inp = (q, k, v, g, beta)
        L, H, d = q.shape
        dev = q.device
        self.cu = torch.tensor([0, L], dtype=torch.int32, device=dev)
        self.L = L
        self.seg = int(segment_len) if segment_len else ((L + 63) // 64) * 64
        self.P = -(-L // self.seg)
        self.pool = final_state.view(1, H, d, d)      # the shard's final state is written here
        self.slots = torch.zeros(1, dtype=torch.int32, device=dev)
        self.out = out
        n = kda_segmented_workspace_size(*self.inp, self.cu, L, self.pool, self.slots, out, self.seg)
        self.ws = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
        self.H, self.d = H, d

    def _args(self):
        return (*self.inp, self.cu, self.L, self.pool, self.slots, self.out)

    def fragments(self):
        """[P, H, d, 2d]: S~ | M of every segment of the shard, in token order."""
        kda_prefill_records(*self._args(), workspace=self.ws)
        frag = torch.empty(1, self.P, self.H, self.d, 2 * self.d, device=self.out.device)
        kda_kcp_fragments(*self._args(), self.seg, self.ws, frag)
        return frag[0]

    def scan(self, frags, s0):
        entries = torch.empty(frags.shape[0], self.H, self.d, self.d, device=frags.device)
        kda_kcp_scan(frags, s0, entries)
        return entries

    def outputs(self, entries):
        """Outputs and the shard's final state from the entry states of its P segments [P, H, d, d]."""
        kda_kcp_outputs(*self._args(), self.seg, self.ws, entries.contiguous().view(1, self.P, self.H, self.d, self.d))


def kcp_prefill(ops, s0, group=None):
    """Runs this rank's part of a sequence-sharded prefill and returns the entry states of all ranks' shards
    [W, H, d, d].  `ops` carries the shard (LibraryOps on a GPU) and returns its segments' fragments
    [P, H, d, 2d] with P equal on every rank; s0 [H, d, d] is the sequence's initial state, the same on
    every rank (or None for zero)."""
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    frag = ops.fragments().contiguous()
    P = frag.shape[0]
    parts = [torch.empty_like(frag) for _ in range(world)]
    dist.all_gather(parts, frag, group=group)
    frags = torch.cat(parts)  # [W * P, H, d, 2d]: rank order, then segment order = token order
    entries = ops.scan(frags, s0)
    ops.outputs(entries[rank * P:(rank + 1) * P])
    return entries[::P]


def shard_bounds(T: int, world: int) -> np.ndarray:
    """Token offsets of `world` contiguous shards of a T-token sequence, as equal as possible (T >= world)."""
    return np.array([(T * r) // world for r in range(world + 1)], np.int64)
