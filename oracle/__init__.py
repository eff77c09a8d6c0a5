"""KDA oracle -- TEST INFRASTRUCTURE ONLY.

Plain fp64 CPU implementation of the KDA recurrence (``kda_oracle.c``), used by
the tests, the smoke check and the benchmark's CPU-baseline leg to judge the
CUDA library.  The product path never imports this package; this package never
imports the CUDA library.  The two share only the seeded input generator
(``synth``), which holds none of the method's arithmetic.

Functions follow these passages:

* ``recurrence`` -- "Kimi K3: architecture and SGLang Day-0 Support", section
  "attention mechanism explained: KDA", math box (gate, read, delta write), and
  the linear-attention section for the read-out o = S^T q after the write.
* ``transition`` -- "Kimi K3 infra report reading", sections 4.1-4.2 (the
  per-token transition M_t = (I - beta k k^T) Diag(alpha) and a segment's
  cumulative transition M, the first KCP fragment).
* ``backward`` -- the vector-Jacobian product of ``recurrence`` (every forward
  line of the KDA math box differentiated in reverse order), the gradient the
  training side of "Kimi K3 infra report reading", section 7, needs.
* ``short_conv_step``, ``fused_decode`` -- the decode token with its short causal convolution in front
  and the gated output norm behind ("SGLang and Miles: day-0 support for Kimi K3", kernels: the fused
  Conv + KDA + Onorm decode kernel; the stages' formulas are this package's reading, see the docstring).
* ``decode``, ``verify``, ``fold`` -- the same recurrence over 1 or W tokens;
  "SGLang and Miles day-0 support for Kimi K3", section "ReplaySSM": verify
  reads the committed state and never writes it, fold replays only the accepted
  prefix from the committed state.

Pins: every function here is checked against closed forms, invariants, the
pages' worked example, brute force and finite differences, in
``tests/test_oracle_pins.py`` (recurrence, transition, decode / verify / fold,
and the packing, snapshot and sampling bookkeeping), ``tests/test_oracle_backward_pins.py``
(backward) and ``tests/test_oracle_fused_pins.py`` (short convolution, fused decode).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None

F32, BF16, F64 = 0, 1, 2

MUTATIONS = {
    "none": 0,
    "no_gate": 1,
    "delta_sign": 2,
    "transposed_read": 3,
    "read_before_write": 4,
    "gate_after_write": 5,
    "no_beta": 6,
    "stale_decay": 7,
}


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc: strict ISO C11, no FMA contraction, no arch flags."""
    src = os.path.join(_HERE, "kda_oracle.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    tmp = _SO + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O3", "-std=c11", "-D_POSIX_C_SOURCE=200809L", "-ffp-contract=off", "-fPIC",
                           "-shared", "-pthread", src, "-o", tmp, "-lm"])
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i32, i64, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
        lib.kda_oracle_default_threads.restype = i32
        lib.kda_oracle_recurrence.restype = i32
        lib.kda_oracle_recurrence.argtypes = [i32, vp, i32, i32, i32, i32, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp,
                                              vp, i64, vp, vp, i32, i32]
        lib.kda_oracle_backward.restype = i32
        lib.kda_oracle_backward.argtypes = [i32, vp, i32, i32, i32, i32, vp, vp, vp, i32, vp, vp, vp, i32, vp, vp,
                                            vp, vp, vp, vp, vp, vp, i32, i32]
        lib.kda_oracle_transition.restype = i32
        lib.kda_oracle_transition.argtypes = [i32, vp, i32, i32, i32, vp, i32, vp, vp, vp, i32]
        _lib = lib
    return _lib


def default_threads() -> int:
    return int(_load().kda_oracle_default_threads())


def _xdtype(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"unsupported input dtype {a.dtype}")


def _gdtype(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"unsupported gate dtype {a.dtype}")


def _ptr(a):
    return None if a is None else a.ctypes.data


def recurrence(q, k, v, g, beta, cu_seqlens, s0=None, want_o=True, sample_t=None, snap_every=0,
               want_final=True, mutation="none", threads=0):
    """Sequential fp64 KDA recurrence over packed sequences.

    q, k: [T, H, dk]; v: [T, H, dv] (float32, bf16 bits as uint16, or float64)
    g: [T, H, dk] log-decay, beta: [T, H] (float32 or float64)
    cu_seqlens: [N+1] token offsets; s0: [N, H, dk, dv] initial states (any float dtype) or None for zero.
    Returns a dict with 'o' [T,H,dv], 'o_samples' [n,H,dv], 's_final' [N,H,dk,dv],
    'snaps' (list per sequence of [m,H,dk,dv]) and 'threads'.
    """
    q, k, v = (np.ascontiguousarray(x) for x in (q, k, v))
    g, beta = np.ascontiguousarray(g), np.ascontiguousarray(beta)
    xd = _xdtype(q)
    if _xdtype(k) != xd or _xdtype(v) != xd:
        raise TypeError("q, k, v must share a dtype")
    gd = _gdtype(g)
    if _gdtype(beta) != gd:
        raise TypeError("g and beta must share a dtype")
    T, H, dk = q.shape
    dv = v.shape[2]
    if k.shape != (T, H, dk) or v.shape[:2] != (T, H) or g.shape != (T, H, dk) or beta.shape != (T, H):
        raise ValueError("shape mismatch")
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, np.int64))
    N = len(cu) - 1
    if cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
        raise ValueError("bad cu_seqlens")
    s0d = None if s0 is None else np.ascontiguousarray(np.asarray(s0, np.float64).reshape(N, H, dk, dv))
    o = np.zeros((T, H, dv), np.float64) if want_o else None
    sidx = osamp = None
    if sample_t is not None:
        sample_t = np.asarray(sample_t, np.int64)
        sidx = np.full(T, -1, np.int64)
        sidx[sample_t] = np.arange(len(sample_t))
        osamp = np.zeros((len(sample_t), H, dv), np.float64)
    s_final = np.zeros((N, H, dk, dv), np.float64) if want_final else None
    snaps = base = None
    lens = np.diff(cu)
    if snap_every > 0:
        counts = lens // snap_every
        base = np.zeros(N, np.int64)
        base[1:] = np.cumsum(counts)[:-1]
        snaps = np.zeros((max(int(counts.sum()), 1), H, dk, dv), np.float64)
    rc = _load().kda_oracle_recurrence(N, cu.ctypes.data, H, dk, dv, xd, q.ctypes.data, k.ctypes.data,
                                       v.ctypes.data, gd, g.ctypes.data, beta.ctypes.data, _ptr(s0d), _ptr(o),
                                       _ptr(sidx), _ptr(osamp), _ptr(s_final), int(snap_every), _ptr(base),
                                       _ptr(snaps), MUTATIONS[mutation], int(threads))
    if rc < 0:
        raise ValueError("oracle rejected its arguments")
    out = {"o": o, "o_samples": osamp, "s_final": s_final, "threads": rc}
    if snap_every > 0:
        out["snaps"] = [snaps[base[i]:base[i] + lens[i] // snap_every] for i in range(N)]
    return out


BACKWARD_MUTATIONS = {
    "none": 0,
    "no_out_grad": 1,
    "no_read_grad": 2,
    "dg_no_alpha": 3,
    "dk_no_read": 4,
    "dbeta_sign": 5,
    "no_gate_carry": 6,
    "dq_pre_write": 7,
}


def backward(q, k, v, g, beta, cu_seqlens, do, s0=None, ds_final=None, mutation="none", threads=0):
    """Gradients of L = sum_t <do_t, o_t> + <ds_final, S_T> through the fp64 recurrence.

    Inputs as for ``recurrence``; do: [T, H, dv] (float32, bf16 bits as uint16, or float64);
    ds_final: [N, H, dk, dv] or None (zero).  Returns a dict of fp64 arrays 'dq', 'dk' [T,H,dk],
    'dv' [T,H,dv], 'dg' [T,H,dk], 'dbeta' [T,H], 'ds0' [N,H,dk,dv] and 'threads'.
    """
    q, k, v, do = (np.ascontiguousarray(x) for x in (q, k, v, do))
    g, beta = np.ascontiguousarray(g), np.ascontiguousarray(beta)
    xd = _xdtype(q)
    if _xdtype(k) != xd or _xdtype(v) != xd:
        raise TypeError("q, k, v must share a dtype")
    gd = _gdtype(g)
    if _gdtype(beta) != gd:
        raise TypeError("g and beta must share a dtype")
    T, H, dk = q.shape
    dv = v.shape[2]
    if (k.shape != (T, H, dk) or v.shape[:2] != (T, H) or g.shape != (T, H, dk) or beta.shape != (T, H)
            or do.shape != (T, H, dv)):
        raise ValueError("shape mismatch")
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, np.int64))
    N = len(cu) - 1
    if cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
        raise ValueError("bad cu_seqlens")
    f64 = lambda x: None if x is None else np.ascontiguousarray(np.asarray(x, np.float64).reshape(N, H, dk, dv))
    s0d, dsd = f64(s0), f64(ds_final)
    out = {"dq": np.zeros((T, H, dk)), "dk": np.zeros((T, H, dk)), "dv": np.zeros((T, H, dv)),
           "dg": np.zeros((T, H, dk)), "dbeta": np.zeros((T, H)), "ds0": np.zeros((N, H, dk, dv))}
    rc = _load().kda_oracle_backward(N, cu.ctypes.data, H, dk, dv, xd, q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                     gd, g.ctypes.data, beta.ctypes.data, _ptr(s0d), _xdtype(do), do.ctypes.data,
                                     _ptr(dsd), *(out[n].ctypes.data for n in ("dq", "dk", "dv", "dg", "dbeta", "ds0")),
                                     BACKWARD_MUTATIONS[mutation], int(threads))
    if rc == -2:
        raise MemoryError("oracle backward ran out of host memory")
    if rc < 0:
        raise ValueError("oracle rejected its arguments")
    out["threads"] = rc
    return out


def transition(k, g, beta, bounds, threads=0):
    """Cumulative transitions M = M_{t1-1} ... M_{t0} for each token range [bounds[s], bounds[s+1]).

    Returns [n_seg, H, dk, dk] fp64.
    """
    k, g, beta = np.ascontiguousarray(k), np.ascontiguousarray(g), np.ascontiguousarray(beta)
    T, H, dk = k.shape
    b = np.ascontiguousarray(np.asarray(bounds, np.int64))
    n = len(b) - 1
    M = np.zeros((max(n, 1), H, dk, dk), np.float64)
    rc = _load().kda_oracle_transition(n, b.ctypes.data, H, dk, _xdtype(k), k.ctypes.data, _gdtype(g),
                                       g.ctypes.data, beta.ctypes.data, M.ctypes.data, int(threads))
    if rc < 0:
        raise ValueError("oracle rejected its arguments")
    return M[:n]


def decode(pool, slot_ids, q, k, v, g, beta, threads=0):
    """One token per request from the committed states pool[slot_ids].

    q, k, g: [B, H, dk]; v: [B, H, dv]; beta: [B, H].  Returns (o [B,H,dv], new states [B,H,dk,dv]).
    """
    B = q.shape[0]
    r = recurrence(q, k, v, g, beta, np.arange(B + 1), s0=pool[np.asarray(slot_ids)], threads=threads)
    return r["o"], r["s_final"]


def verify(pool, slot_ids, wq, wk, wv, wg, wbeta, threads=0):
    """Draft window of W tokens per request from the committed states (which it leaves untouched).

    w*: [B, W, H, .].  Returns (o [B,W,H,dv], states after each window token [B,W,H,dk,dv]).
    """
    B, W = wq.shape[:2]
    flat = lambda x: np.ascontiguousarray(x.reshape((B * W,) + x.shape[2:]))
    r = recurrence(flat(wq), flat(wk), flat(wv), flat(wg), flat(wbeta), np.arange(0, B * W + 1, W),
                   s0=pool[np.asarray(slot_ids)], snap_every=1, threads=threads)
    o = r["o"].reshape((B, W) + r["o"].shape[1:])
    states = np.stack(r["snaps"])  # [B, W, H, dk, dv]
    return o, states


def fold(pool, slot_ids, wq, wk, wv, wg, wbeta, accepted, threads=0):
    """Committed states after replaying the accepted prefix (n = accepted[b] tokens) of each window.

    Requests with n = 0 keep their committed state.  Returns [B, H, dk, dv] fp64.
    """
    _, states = verify(pool, slot_ids, wq, wk, wv, wg, wbeta, threads=threads)
    committed = np.asarray(pool[np.asarray(slot_ids)], np.float64)
    out = committed.copy()
    for b, n in enumerate(np.asarray(accepted)):
        if n > 0:
            out[b] = states[b, n - 1]
    return out


# ------------------------------------------------------------------ fused decode front/back-end

G_MIN = -5.0     # lower bound of the log-decay
CONV_WIDTH = 4   # taps of the short causal convolution
L2_EPS = 1e-6    # inside the square root of the q / k normalisation


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def _widen(x):
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def short_conv_step(x, conv_state, w):
    """One token of a depthwise causal convolution followed by SiLU.

    x [..., C] the token's input; conv_state [..., C, W-1] the previous W-1 inputs, oldest first;
    w [C, W] the taps, w[c, W-1] multiplying the current input.  Returns (SiLU(y), new state) with
    y_c = sum_tau w[c, tau] * window[c, tau] over the window (state, x).
    """
    window = np.concatenate([conv_state, x[..., None]], axis=-1)
    y = (window * w).sum(axis=-1)
    return y * _sigmoid(y), window[..., 1:]


def fused_decode(pool, conv_state, slot_ids, xq, xk, xv, a, b, z, conv_w, norm_w, eps, threads=0):
    """One decode token per request through the short convolution, the KDA step and the gated output norm.

    The pages print no formula for the convolution, the normalisations or the gates; what follows is the
    plainest reading, pinned by its properties (stepwise = full causal convolution, the read-back identity
    through the composed path, unit rms and scale invariance of the output norm, the gates' limits and
    midpoints checked through the state and the output) rather than by a second copy of the expressions.
    Reading of "SGLang and Miles: day-0 support for Kimi K3" (kernels: the fused Conv + KDA + Onorm decode
    kernel), "Kimi K3: Architecture and SGLang Day-0 Support" (KDA math box: the log-decay kept above
    g_min = -5 by a scaled sigmoid; the output gate a full-rank projection of the input) and "Kimi K3
    infra report reading" section 7 (the recurrent state and the conv edges are the two carried parts):
      q, k, v = SiLU(causal conv_4(x_q, x_k, x_v))           (per channel, window = 3 carried inputs + x)
      q, k    = q / sqrt(|q|^2 + 1e-6), k / sqrt(|k|^2 + 1e-6)
      g = G_MIN * sigmoid(a),  beta = sigmoid(b)
      o = the KDA step (``recurrence`` over one token) from pool[slot]
      y = o / sqrt(mean(o^2) + eps) * norm_w * sigmoid(z)
    xq, xk, xv, z [B, H, d] (fp32, bf16 bits or fp64), a [B, H, dk], b [B, H]; pool [S, H, dk, dv];
    conv_state [S, H, 3, W-1, d] (streams q, k, v; taps oldest first); conv_w [3, H, d, W]; norm_w [dv].
    Returns (y [B, H, dv], new states [B, H, dk, dv], new conv states [B, H, 3, W-1, d]) in fp64.
    """
    slot_ids = np.asarray(slot_ids)
    xs = [_widen(t) for t in (xq, xk, xv)]
    cs = _widen(conv_state)[slot_ids]                  # [B, H, 3, W-1, d]
    cw = _widen(conv_w)                                # [3, H, d, W]
    outs, new_cs = [], np.empty_like(cs)
    for s in range(3):
        st = np.moveaxis(cs[:, :, s], -2, -1)         # [B, H, d, W-1]
        y, nst = short_conv_step(xs[s], st, cw[s])    # w [H, d, W] broadcasts over B
        outs.append(y)
        new_cs[:, :, s] = np.moveaxis(nst, -1, -2)
    q, k, v = outs
    q = q / np.sqrt((q * q).sum(-1, keepdims=True) + L2_EPS)
    k = k / np.sqrt((k * k).sum(-1, keepdims=True) + L2_EPS)
    g = G_MIN * _sigmoid(_widen(a))
    beta = _sigmoid(_widen(b))
    B = q.shape[0]
    r = recurrence(q, k, v, g, beta, np.arange(B + 1), s0=_widen(pool)[slot_ids], threads=threads)
    o = r["o"]
    y = o / np.sqrt((o * o).mean(-1, keepdims=True) + eps) * _widen(norm_w) * _sigmoid(_widen(z))
    return y, r["s_final"], new_cs
