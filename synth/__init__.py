"""Seeded synthetic inputs for the KDA workloads.

This module is shared by the tests, the benchmark and the oracle harness.  It
draws random numbers (counter-based SplitMix64 + Box-Muller, implemented in
``synth.c``) and shapes them into the input distributions of the five
workloads; it contains none of the KDA recurrence's arithmetic.

Workloads (all sizes are the defaults; tests shrink them through keyword
arguments):

1. ``tiny``        1 sequence, T=64, H=2, dk=dv=16, fp32 inputs, zero initial state.
2. ``prefill_8k``  B=1, T=8192, H=12, d=128, bf16 q/k/v, S0 ~ N(0, 0.02).
3. ``varlen``      16 sequences, lengths round(exp(U(ln 512, ln 32768))), a
                   256-slot state pool, distinct random slots, snapshots every
                   4 chunks into a ping-pong extra pool.
4. ``decode_verify`` 256 requests in a 1024-slot pool, one decode token, then an
                   8-token draft window with accepted length min(Poisson(2.7), 8).
5. ``long_1m``     B=1, T=1,048,576, H=12, d=128, 64 segments of 16,384 tokens,
                   4096 sampled output positions.

q and k rows are N(0,1) then L2-normalised per (token, head) in fp64; v is N(0,1);
beta = sigmoid(N(0,1)); the log-decay g = ln(alpha) = -softplus(N(mean,1)) * scale
clamped at -5 (mean=-2, scale=1 for d=128 workloads; mean=0, scale=0.1 for tiny).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_build", "libsynth.so")
_lib = None

F32, BF16, F64 = 0, 1, 2
G_MIN = -5.0

# stream ids (one per array kind)
S_Q, S_K, S_V, S_G, S_BETA, S_S0 = 1, 2, 3, 4, 5, 6
S_LEN, S_SLOTS, S_ACCEPT, S_SAMPLES, S_EXTRA = 7, 8, 9, 10, 11
S_WQ, S_WK, S_WV, S_WG, S_WBETA = 21, 22, 23, 24, 25
S_DO, S_DFINAL = 31, 32
S_FX, S_FA, S_FB, S_FZ, S_FCS, S_FCW, S_FNW = 41, 42, 43, 44, 45, 46, 47


def build(force: bool = False) -> str:
    """Compile libsynth.so with gcc (plain C, no architecture-specific flags)."""
    src = os.path.join(_HERE, "synth.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    tmp = _SO + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", src, "-o", tmp, "-lm"])
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, i32, f64, vp = ctypes.c_uint64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        lib.synth_draw.restype = u64
        lib.synth_draw.argtypes = [u64, u64, u64]
        lib.synth_uniform.restype = f64
        lib.synth_uniform.argtypes = [u64, u64, u64]
        lib.synth_normal.restype = f64
        lib.synth_normal.argtypes = [u64, u64, u64]
        lib.synth_normal_fill.argtypes = [u64, u64, u64, f64, f64, i32, vp, i32]
        lib.synth_uniform_fill.argtypes = [u64, u64, u64, vp, i32]
        lib.synth_unit_rows.restype = i32
        lib.synth_unit_rows.argtypes = [u64, u64, u64, i32, i32, vp, i32]
        lib.synth_log_decay.argtypes = [u64, u64, u64, f64, f64, f64, vp, i32]
        lib.synth_sigmoid_normal.argtypes = [u64, u64, u64, vp, i32]
        _lib = lib
    return _lib


_NP = {F32: np.float32, BF16: np.uint16, F64: np.float64}


def draw(seed: int, stream: int, i: int) -> int:
    return int(_load().synth_draw(seed, stream, i))


def uniform(seed: int, stream: int, n: int, threads: int = 0) -> np.ndarray:
    out = np.empty(n, np.float64)
    _load().synth_uniform_fill(seed, stream, n, out.ctypes.data, threads)
    return out


def normal(seed: int, stream: int, shape, mean=0.0, std=1.0, dtype=F32, threads: int = 0) -> np.ndarray:
    out = np.empty(shape, _NP[dtype])
    _load().synth_normal_fill(seed, stream, out.size, mean, std, dtype, out.ctypes.data, threads)
    return out


def unit_rows(seed: int, stream: int, shape, dtype=F32, threads: int = 0) -> np.ndarray:
    """Rows along the last axis are N(0,1) vectors normalised to unit L2 norm (fp64), then rounded."""
    out = np.empty(shape, _NP[dtype])
    d = shape[-1]
    rc = _load().synth_unit_rows(seed, stream, out.size // d, d, dtype, out.ctypes.data, threads)
    if rc != 0:
        raise ValueError("unit_rows: row length out of range")
    return out


def log_decay(seed: int, stream: int, shape, mean=-2.0, scale=1.0, floor=G_MIN, threads: int = 0) -> np.ndarray:
    out = np.empty(shape, np.float32)
    _load().synth_log_decay(seed, stream, out.size, mean, scale, floor, out.ctypes.data, threads)
    return out


def sigmoid_normal(seed: int, stream: int, shape, threads: int = 0) -> np.ndarray:
    out = np.empty(shape, np.float32)
    _load().synth_sigmoid_normal(seed, stream, out.size, out.ctypes.data, threads)
    return out


def bf16_to_f32(x: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 exactly."""
    return (x.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 bit patterns (round to nearest even)."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def distinct_slots(seed: int, stream: int, n: int, num_slots: int) -> np.ndarray:
    """n distinct slot ids drawn uniformly from [0, num_slots) (a random permutation prefix)."""
    if n > num_slots:
        raise ValueError("more slots requested than the pool holds")
    perm = np.argsort(uniform(seed, stream, num_slots), kind="stable")
    return perm[:n].astype(np.int32)


def poisson_clipped(seed: int, stream: int, n: int, lam: float, hi: int) -> np.ndarray:
    """min(Poisson(lam), hi) by inverse-CDF on one uniform per draw."""
    u = uniform(seed, stream, n)
    out = np.empty(n, np.int32)
    for i, ui in enumerate(u):
        k, p = 0, math.exp(-lam)
        cdf = p
        while ui > cdf and k < hi:
            k += 1
            p *= lam / k
            cdf += p
        out[i] = k
    return out


@dataclass
class Prefill:
    """A packed varlen prefill problem: token-major inputs and a slot-indexed state pool."""
    name: str
    seed: int
    H: int
    dk: int
    dv: int
    in_dtype: int                 # F32 or BF16 for q, k, v
    q: np.ndarray                 # [T, H, dk]
    k: np.ndarray                 # [T, H, dk]
    v: np.ndarray                 # [T, H, dv]
    g: np.ndarray                 # [T, H, dk] fp32, log-decay
    beta: np.ndarray              # [T, H] fp32
    cu_seqlens: np.ndarray        # [N+1] int32
    pool: np.ndarray              # [num_slots, H, dk, dv] fp32
    slot_ids: np.ndarray          # [N] int32
    init_zero: bool
    extra_pool: np.ndarray | None = None      # [num_extra, H, dk, dv] fp32
    extra_slot_ids: np.ndarray | None = None  # [N, 2] int32
    snapshot_every_chunks: int = 0
    segment_len: int = 0
    sample_t: np.ndarray | None = None        # sampled global token positions (sorted)
    meta: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def N(self) -> int:
        return len(self.cu_seqlens) - 1

    @property
    def lengths(self) -> np.ndarray:
        return np.diff(self.cu_seqlens.astype(np.int64))


def _tokens(seed, T, H, dk, dv, dtype, g_mean, g_scale, threads, g_floor=G_MIN):
    q = unit_rows(seed, S_Q, (T, H, dk), dtype, threads)
    k = unit_rows(seed, S_K, (T, H, dk), dtype, threads)
    v = normal(seed, S_V, (T, H, dv), dtype=dtype, threads=threads)
    g = log_decay(seed, S_G, (T, H, dk), g_mean, g_scale, g_floor, threads)
    beta = sigmoid_normal(seed, S_BETA, (T, H), threads)
    return q, k, v, g, beta


def tiny(seed: int = 1, T: int = 64, H: int = 2, d: int = 16, threads: int = 0) -> Prefill:
    q, k, v, g, beta = _tokens(seed, T, H, d, d, F32, 0.0, 0.1, threads)
    return Prefill("tiny", seed, H, d, d, F32, q, k, v, g, beta,
                   np.array([0, T], np.int32), np.zeros((1, H, d, d), np.float32),
                   np.array([0], np.int32), init_zero=True)


def prefill_8k(seed: int = 2, T: int = 8192, H: int = 12, d: int = 128, dtype: int = BF16,
               threads: int = 0) -> Prefill:
    q, k, v, g, beta = _tokens(seed, T, H, d, d, dtype, -2.0, 1.0, threads)
    pool = normal(seed, S_S0, (1, H, d, d), 0.0, 0.02, F32, threads)
    return Prefill("prefill_8k", seed, H, d, d, dtype, q, k, v, g, beta,
                   np.array([0, T], np.int32), pool, np.array([0], np.int32), init_zero=False)


def varlen_lengths(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    u = uniform(seed, S_LEN, n)
    return np.rint(np.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))).astype(np.int64)


def varlen(seed: int = 3, n_seqs: int = 16, lo: int = 512, hi: int = 32768, H: int = 12, d: int = 128,
           num_slots: int = 256, num_extra: int = 64, snapshot_every_chunks: int = 4, dtype: int = BF16,
           lengths=None, threads: int = 0) -> Prefill:
    lens = np.asarray(lengths, np.int64) if lengths is not None else varlen_lengths(seed, n_seqs, lo, hi)
    n_seqs = len(lens)
    cu = np.zeros(n_seqs + 1, np.int64)
    cu[1:] = np.cumsum(lens)
    T = int(cu[-1])
    q, k, v, g, beta = _tokens(seed, T, H, d, d, dtype, -2.0, 1.0, threads)
    pool = normal(seed, S_S0, (num_slots, H, d, d), 0.0, 0.02, F32, threads)
    slots = distinct_slots(seed, S_SLOTS, n_seqs, num_slots)
    extra_slots = distinct_slots(seed, S_EXTRA, 2 * n_seqs, num_extra).reshape(n_seqs, 2)
    extra_pool = np.zeros((num_extra, H, d, d), np.float32)
    return Prefill("varlen", seed, H, d, d, dtype, q, k, v, g, beta, cu.astype(np.int32), pool, slots,
                   init_zero=False, extra_pool=extra_pool, extra_slot_ids=extra_slots,
                   snapshot_every_chunks=snapshot_every_chunks)


def long_1m(seed: int = 5, T: int = 1 << 20, H: int = 12, d: int = 128, segment_len: int = 16384,
            n_samples: int = 4096, dtype: int = BF16, threads: int = 0) -> Prefill:
    q, k, v, g, beta = _tokens(seed, T, H, d, d, dtype, -2.0, 1.0, threads)
    pool = normal(seed, S_S0, (1, H, d, d), 0.0, 0.02, F32, threads)
    n_samples = min(n_samples, T)
    samp = np.sort(np.argsort(uniform(seed, S_SAMPLES, T), kind="stable")[:n_samples]).astype(np.int64)
    return Prefill("long_1m", seed, H, d, d, dtype, q, k, v, g, beta, np.array([0, T], np.int32), pool,
                   np.array([0], np.int32), init_zero=False, segment_len=segment_len, sample_t=samp)


def output_grads(prob: Prefill, seed: int):
    """Seeded upstream gradients for a backward pass over `prob`: dL/do [T, H, dv] N(0, 1) in the input
    dtype and dL/dS_T [N, H, dk, dv] N(0, 0.1) fp32."""
    d_out = normal(seed, S_DO, (prob.T, prob.H, prob.dv), dtype=prob.in_dtype)
    d_final = normal(seed, S_DFINAL, (prob.N, prob.H, prob.dk, prob.dv), 0.0, 0.1, F32)
    return d_out, d_final


def fused_decode_inputs(seed: int, B: int, H: int, d: int, num_slots: int, steps: int = 1, dtype: int = BF16,
                        with_pool: bool = True, threads: int = 0) -> dict:
    """Seeded inputs of `steps` consecutive fused decode tokens for B requests: pre-convolution projections
    xq, xk, xv [steps, B, H, d] N(0, 1) and output-gate logits z (input dtype); decay logits a [steps, B, H, d]
    and write-strength logits b [steps, B, H] N(0, 1) fp32; carried convolution inputs
    [num_slots, H, 3, 3, d] N(0, 1), taps [3, H, d, 4] N(0, 0.5), norm weight [d] U(0.5, 1.5) (fp32); a state
    pool [num_slots, H, d, d] N(0, 0.02) (None without with_pool) and B distinct slots."""
    x = normal(seed, S_FX, (3, steps, B, H, d), dtype=dtype, threads=threads)
    return dict(xq=x[0], xk=x[1], xv=x[2],
                a=normal(seed, S_FA, (steps, B, H, d), threads=threads),
                b=normal(seed, S_FB, (steps, B, H), threads=threads),
                z=normal(seed, S_FZ, (steps, B, H, d), dtype=dtype, threads=threads),
                conv_state=normal(seed, S_FCS, (num_slots, H, 3, 3, d), threads=threads),
                conv_w=normal(seed, S_FCW, (3, H, d, 4), 0.0, 0.5, threads=threads),
                norm_w=(0.5 + uniform(seed, S_FNW, d)).astype(np.float32),
                pool=normal(seed, S_S0, (num_slots, H, d, d), 0.0, 0.02, F32, threads) if with_pool else None,
                slot_ids=distinct_slots(seed, S_SLOTS, B, num_slots))


@dataclass
class DecodeVerify:
    """Batched decode token + speculative window over a slot-indexed pool."""
    seed: int
    B: int
    W: int
    H: int
    dk: int
    dv: int
    in_dtype: int
    pool: np.ndarray          # [num_slots, H, dk, dv] fp32
    slot_ids: np.ndarray      # [B] int32, distinct
    # decode token, [B, H, .]
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    g: np.ndarray
    beta: np.ndarray
    # draft window, [B, W, H, .]
    wq: np.ndarray
    wk: np.ndarray
    wv: np.ndarray
    wg: np.ndarray
    wbeta: np.ndarray
    accepted: np.ndarray      # [B] int32 in [0, W]


def decode_verify(seed: int = 4, B: int = 256, W: int = 8, H: int = 12, d: int = 128, num_slots: int = 1024,
                  mean_accept: float = 2.7, dtype: int = BF16, threads: int = 0) -> DecodeVerify:
    pool = normal(seed, S_S0, (num_slots, H, d, d), 0.0, 0.02, F32, threads)
    slots = distinct_slots(seed, S_SLOTS, B, num_slots)
    q = unit_rows(seed, S_Q, (B, H, d), dtype, threads)
    k = unit_rows(seed, S_K, (B, H, d), dtype, threads)
    v = normal(seed, S_V, (B, H, d), dtype=dtype, threads=threads)
    g = log_decay(seed, S_G, (B, H, d), -2.0, 1.0, G_MIN, threads)
    beta = sigmoid_normal(seed, S_BETA, (B, H), threads)
    wq = unit_rows(seed, S_WQ, (B, W, H, d), dtype, threads)
    wk = unit_rows(seed, S_WK, (B, W, H, d), dtype, threads)
    wv = normal(seed, S_WV, (B, W, H, d), dtype=dtype, threads=threads)
    wg = log_decay(seed, S_WG, (B, W, H, d), -2.0, 1.0, G_MIN, threads)
    wbeta = sigmoid_normal(seed, S_WBETA, (B, W, H), threads)
    acc = poisson_clipped(seed, S_ACCEPT, B, mean_accept, W)
    return DecodeVerify(seed, B, W, H, d, d, dtype, pool, slots, q, k, v, g, beta, wq, wk, wv, wg, wbeta, acc)
