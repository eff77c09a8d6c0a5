"""KCP across ranks: the host-side exchange of kcp_prefill, run as two gloo processes on the CPU.

Each rank holds one contiguous shard of a sequence.  The per-rank compute is done by the fp64 oracle here
(the fragment: the shard's state from a zero input state and its cumulative transition; the outputs: the
recurrence from the entry state); the exchange, its rank order and the entry selection are the library's
kcp_prefill.  Every rank's outputs and the last rank's final state must equal the unsplit recurrence, and
all ranks must hold identical entry states.
"""
import os
import socket
import sys

import numpy as np
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _problem():
    rng = np.random.default_rng(21)
    T, H, d = 150, 2, 8
    k = rng.standard_normal((T, H, d))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    return dict(q=rng.standard_normal((T, H, d)), k=k, v=rng.standard_normal((T, H, d)),
                g=-np.abs(rng.standard_normal((T, H, d))) * 0.3, beta=rng.uniform(0.05, 0.95, (T, H))), \
        rng.standard_normal((H, d, d)) * 0.1


class OracleOps:
    """The per-rank compute of KCP by the fp64 oracle (test stand-in for the GPU kernels), with the shard cut
    into segments of `seg` tokens like LibraryOps."""

    def __init__(self, shard, seg):
        self.shard = shard
        L = shard["q"].shape[0]
        self.bounds = list(range(0, L, seg)) + [L]
        self.out = self.final = None

    def _seg(self, p):
        return {n: x[self.bounds[p]:self.bounds[p + 1]] for n, x in self.shard.items()}

    def fragments(self):
        import oracle
        out = []
        for p in range(len(self.bounds) - 1):
            s = self._seg(p)
            L = s["q"].shape[0]
            zero = oracle.recurrence(s["q"], s["k"], s["v"], s["g"], s["beta"], [0, L])["s_final"][0]
            M = oracle.transition(s["k"], s["g"], s["beta"], [0, L])[0]
            out.append(np.concatenate([zero, M], axis=-1))  # [H, d, 2d]: S~ | M
        return torch.from_numpy(np.stack(out))

    def scan(self, frags, s0):
        f = frags.numpy()
        d = f.shape[2]
        e = [np.zeros_like(f[0, :, :, :d]) if s0 is None else s0.numpy()]
        for p in range(f.shape[0] - 1):
            e.append(np.einsum("hij,hjc->hic", f[p, :, :, d:], e[-1]) + f[p, :, :, :d])
        return torch.from_numpy(np.stack(e))

    def outputs(self, entries):
        import oracle
        outs = []
        for p in range(len(self.bounds) - 1):  # each segment from its own entry state
            s = self._seg(p)
            r = oracle.recurrence(s["q"], s["k"], s["v"], s["g"], s["beta"], [0, s["q"].shape[0]],
                                  s0=entries[p].numpy()[None])
            outs.append(r["o"])
            self.final = r["s_final"][0]
        self.out = np.concatenate(outs)


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    from kda_gated_delta_rule_gb300.kcp import kcp_prefill, kcp_segment_len, shard_bounds

    dist.init_process_group("gloo", rank=rank, world_size=world)
    full, s0 = _problem()
    T = full["q"].shape[0]
    b = shard_bounds(T, world)
    seg = kcp_segment_len(T, world, 3)  # 75-token shards: two segments of 64 and 11 tokens each
    ops = OracleOps({n: x[b[rank]:b[rank + 1]] for n, x in full.items()}, seg)
    entries = kcp_prefill(ops, torch.from_numpy(s0))
    q.put((rank, entries.numpy(), ops.out, ops.final))
    dist.destroy_process_group()


def test_two_ranks_reproduce_the_unsplit_recurrence():
    import oracle
    from kda_gated_delta_rule_gb300.kcp import shard_bounds

    world = 2
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    full, s0 = _problem()
    T = full["q"].shape[0]
    ref = oracle.recurrence(*(full[n] for n in ("q", "k", "v", "g", "beta")), [0, T], s0=s0[None])
    b = shard_bounds(T, world)
    np.testing.assert_array_equal(res[0][1], res[1][1])  # identical entry states on every rank
    for rank, entries, out, final in res:
        np.testing.assert_allclose(out, ref["o"][b[rank]:b[rank + 1]], rtol=0, atol=1e-11)
    np.testing.assert_allclose(res[-1][3], ref["s_final"][0], rtol=0, atol=1e-11)
    # the scan's entry state of rank 1 is the state after rank 0's tokens
    head = oracle.recurrence(*(full[n][:b[1]] for n in ("q", "k", "v", "g", "beta")), [0, b[1]], s0=s0[None])
    np.testing.assert_allclose(res[0][1][1], head["s_final"][0], rtol=0, atol=1e-11)


def test_shard_bounds_cover_the_sequence_evenly():
    """Contiguous shards in rank order that cover [0, T) exactly, none empty, sizes within one token."""
    sys.path.insert(0, ROOT)
    from kda_gated_delta_rule_gb300.kcp import shard_bounds
    for T in (1, 7, 150, 8192, 1_048_579):
        for world in range(1, 9):
            if T < world:
                continue
            b = shard_bounds(T, world)
            sizes = np.diff(b)
            assert len(b) == world + 1 and b[0] == 0 and b[-1] == T
            assert sizes.min() >= 1 and sizes.max() - sizes.min() <= 1


def test_common_segment_length_gives_every_rank_the_same_count():
    sys.path.insert(0, ROOT)
    from kda_gated_delta_rule_gb300.kcp import kcp_segment_len, shard_bounds
    for T in (150, 8192, 8193, 64 * 24 + 1, 1 << 20, 1_048_579):
        for world in (1, 2, 3, 8):
            for per_rank in (1, 3, 12):
                seg = kcp_segment_len(T, world, per_rank)
                assert seg % 64 == 0
                counts = {-(-int(n) // seg) for n in np.diff(shard_bounds(T, world))}
                assert len(counts) == 1
