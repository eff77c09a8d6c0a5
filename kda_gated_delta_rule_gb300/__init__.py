"""Python binding of the KDA CUDA library (libkda.so, C ABI in include/kda.h).

Argument marshalling only: every function checks its tensors' shapes and dtypes against the layouts the
header states, passes their device pointers and the current CUDA stream to the C entry point of the same
name, and raises KdaError on a non-OK status.  There is no CPU fallback: if the library is not built,
every call fails.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

__all__ = [
    "KdaError", "load", "lib_path", "KDA_OK", "KDA_DEV_SLOT_OOB", "KDA_DEV_SEQ_OOB", "KDA_DEV_TIMEOUT",
    "KDA_DEV_ACCEPT_OOB", "kda_status_string", "kda_version", "kda_state_bytes_per_head", "kda_state_copy",
    "kda_decode_step", "kda_replay_bytes", "kda_verify", "kda_verify_replay", "kda_prefill_varlen",
    "kda_prefill_workspace_size", "kda_prefill_segmented", "kda_segmented_workspace_size",
    "kda_segment_fragments", "kda_fragment_scan", "kda_segment_outputs", "kda_prefill_segmented_noalloc",
    "kda_prefill_records", "kda_prefill_chain", "kda_cfbi_cache_bytes_per_head", "kda_cfbi_prefill",
    "kda_cfbi_prefill_chunked_workspace_size", "kda_cfbi_prefill_chunked",
    "kda_cfbi_decode", "kda_backward_workspace_size", "kda_prefill_backward", "kda_fused_decode",
    "kda_kcp_fragments", "kda_kcp_scan", "kda_kcp_outputs", "kda_check_slot_ids", "kda_set_debug_checks",
    "kda_debug_checks", "kda_set_test_fault", "KDA_TEST_FAULT_NONE", "KDA_TEST_FAULT_STALL_RECORD_INPUTS", "CFBI_CHUNK", "CFBI_ROW_FLOATS", "EXPORTED_SYMBOLS",
]

KDA_OK = 0
KDA_TEST_FAULT_NONE, KDA_TEST_FAULT_STALL_RECORD_INPUTS = 0, 1
KDA_DEV_SLOT_OOB, KDA_DEV_SEQ_OOB, KDA_DEV_TIMEOUT, KDA_DEV_ACCEPT_OOB = 1, 2, 4, 8
F32, BF16 = 0, 1
CFBI_CHUNK, CFBI_ROW_FLOATS = 16, 420  # KDA_CFBI_CHUNK, KDA_CFBI_ROW_FLOATS

# every function include/kda.h declares
EXPORTED_SYMBOLS = (
    "kda_status_string", "kda_version", "kda_state_bytes_per_head", "kda_prefill_args_bytes", "kda_state_copy",
    "kda_decode_step", "kda_replay_bytes", "kda_verify", "kda_verify_replay", "kda_prefill_varlen",
    "kda_prefill_workspace_size", "kda_prefill_segmented", "kda_segmented_workspace_size",
    "kda_segment_fragments", "kda_fragment_scan", "kda_segment_outputs", "kda_prefill_segmented_noalloc",
    "kda_prefill_records", "kda_prefill_chain", "kda_cfbi_cache_bytes_per_head", "kda_cfbi_prefill",
    "kda_cfbi_prefill_chunked_workspace_size", "kda_cfbi_prefill_chunked",
    "kda_cfbi_decode", "kda_backward_args_bytes", "kda_backward_workspace_size", "kda_prefill_backward",
    "kda_fused_decode_args_bytes", "kda_fused_decode", "kda_kcp_fragments", "kda_kcp_scan", "kda_kcp_outputs",
    "kda_check_slot_ids", "kda_set_debug_checks", "kda_debug_checks", "kda_set_test_fault",
)


class KdaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {kda_status_string(code)} ({code})")
        self.code = code


class PrefillArgs(ctypes.Structure):
    """Mirror of kda_prefill_args."""
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("g", ctypes.c_void_p),
        ("beta", ctypes.c_void_p), ("in_dtype", ctypes.c_int), ("T", ctypes.c_int64), ("H", ctypes.c_int),
        ("dk", ctypes.c_int), ("dv", ctypes.c_int), ("N", ctypes.c_int), ("cu_seqlens", ctypes.c_void_p),
        ("max_seqlen", ctypes.c_int32), ("pool", ctypes.c_void_p), ("num_slots", ctypes.c_int32),
        ("slot_ids", ctypes.c_void_p), ("init_zero", ctypes.c_int), ("out", ctypes.c_void_p),
        ("out_dtype", ctypes.c_int), ("extra_pool", ctypes.c_void_p), ("num_extra_slots", ctypes.c_int32),
        ("extra_slot_ids", ctypes.c_void_p), ("snapshot_every_chunks", ctypes.c_int32),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t), ("dev_status", ctypes.c_void_p),
    ]


class BackwardArgs(ctypes.Structure):
    """Mirror of kda_backward_args."""
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("g", ctypes.c_void_p),
        ("beta", ctypes.c_void_p), ("in_dtype", ctypes.c_int), ("T", ctypes.c_int64), ("H", ctypes.c_int),
        ("dk", ctypes.c_int), ("dv", ctypes.c_int), ("N", ctypes.c_int), ("cu_seqlens", ctypes.c_void_p),
        ("max_seqlen", ctypes.c_int32), ("pool", ctypes.c_void_p), ("num_slots", ctypes.c_int32),
        ("slot_ids", ctypes.c_void_p), ("init_zero", ctypes.c_int), ("d_out", ctypes.c_void_p),
        ("d_final", ctypes.c_void_p), ("dq", ctypes.c_void_p), ("dk_out", ctypes.c_void_p),
        ("dv_out", ctypes.c_void_p), ("dg", ctypes.c_void_p), ("dbeta", ctypes.c_void_p),
        ("d_init", ctypes.c_void_p), ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("dev_status", ctypes.c_void_p),
    ]


class FusedDecodeArgs(ctypes.Structure):
    """Mirror of kda_fused_decode_args."""
    _fields_ = [
        ("xq", ctypes.c_void_p), ("xk", ctypes.c_void_p), ("xv", ctypes.c_void_p), ("a", ctypes.c_void_p),
        ("b", ctypes.c_void_p), ("z", ctypes.c_void_p), ("in_dtype", ctypes.c_int), ("B", ctypes.c_int),
        ("H", ctypes.c_int), ("dk", ctypes.c_int), ("dv", ctypes.c_int), ("pool", ctypes.c_void_p),
        ("num_slots", ctypes.c_int32), ("slot_ids", ctypes.c_void_p), ("conv_state", ctypes.c_void_p),
        ("conv_w", ctypes.c_void_p), ("norm_w", ctypes.c_void_p), ("norm_eps", ctypes.c_float),
        ("out", ctypes.c_void_p), ("out_dtype", ctypes.c_int), ("dev_status", ctypes.c_void_p),
    ]


_lib = None


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Loads libkda.so; raises if it is not built (no fallback path exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        if not build_if_missing:
            raise RuntimeError(f"KDA CUDA library not built ({_build.LIB}); run __graft_entry__.build()")
        _build.build()
    lib = ctypes.CDLL(_build.LIB)
    vp, i32, i64, sz, c_int = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int
    sig = {
        "kda_status_string": (ctypes.c_char_p, [c_int]),
        "kda_version": (c_int, []),
        "kda_state_bytes_per_head": (sz, [c_int, c_int]),
        "kda_prefill_args_bytes": (sz, []),
        "kda_state_copy": (c_int, [vp, i32, vp, vp, i32, vp, i32, i64, vp, vp]),
        "kda_decode_step": (c_int, [vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int, vp, i32, vp, vp, c_int,
                                    vp, vp]),
        "kda_replay_bytes": (sz, [c_int, c_int, c_int, c_int, c_int, c_int]),
        "kda_verify": (c_int, [vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int, c_int, vp, i32, vp, vp, c_int,
                               vp, sz, vp, vp, vp]),
        "kda_verify_replay": (c_int, [vp, i32, vp, c_int, c_int, c_int, c_int, c_int, c_int, vp, sz, vp, vp, vp]),
        "kda_prefill_varlen": (c_int, [ctypes.POINTER(PrefillArgs), vp]),
        "kda_prefill_workspace_size": (sz, [ctypes.POINTER(PrefillArgs)]),
        "kda_prefill_segmented": (c_int, [ctypes.POINTER(PrefillArgs), i32, vp]),
        "kda_segmented_workspace_size": (sz, [ctypes.POINTER(PrefillArgs), i32]),
        "kda_segment_fragments": (c_int, [ctypes.POINTER(PrefillArgs), i32, vp]),
        "kda_fragment_scan": (c_int, [ctypes.POINTER(PrefillArgs), i32, vp]),
        "kda_segment_outputs": (c_int, [ctypes.POINTER(PrefillArgs), i32, vp]),
        "kda_prefill_segmented_noalloc": (c_int, [ctypes.POINTER(PrefillArgs), i32, vp]),
        "kda_prefill_records": (c_int, [ctypes.POINTER(PrefillArgs), vp]),
        "kda_prefill_chain": (c_int, [ctypes.POINTER(PrefillArgs), vp]),
        "kda_cfbi_cache_bytes_per_head": (sz, [c_int, c_int]),
        "kda_cfbi_prefill": (c_int, [vp, vp, vp, vp, vp, vp, i32, i64, i32, c_int, c_int, c_int, c_int, vp, vp, vp,
                                     i32, vp, vp, c_int, vp, vp]),
        "kda_cfbi_prefill_chunked_workspace_size": (sz, [i64, i32, c_int, c_int, c_int]),
        "kda_cfbi_prefill_chunked": (c_int, [vp, vp, vp, vp, vp, vp, i32, i64, i32, c_int, c_int, c_int, c_int, vp,
                                             vp, vp, i32, vp, vp, c_int, vp, sz, vp, vp]),
        "kda_cfbi_decode": (c_int, [vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int, vp, vp, vp, i32, vp, vp,
                                    c_int, vp, vp]),
        "kda_backward_args_bytes": (sz, []),
        "kda_backward_workspace_size": (sz, [ctypes.POINTER(BackwardArgs)]),
        "kda_prefill_backward": (c_int, [ctypes.POINTER(BackwardArgs), vp]),
        "kda_fused_decode_args_bytes": (sz, []),
        "kda_fused_decode": (c_int, [ctypes.POINTER(FusedDecodeArgs), vp]),
        "kda_kcp_fragments": (c_int, [ctypes.POINTER(PrefillArgs), i32, vp, vp]),
        "kda_kcp_scan": (c_int, [vp, i32, c_int, c_int, c_int, vp, vp, vp, vp]),
        "kda_kcp_outputs": (c_int, [ctypes.POINTER(PrefillArgs), i32, vp, vp]),
        "kda_check_slot_ids": (c_int, [vp, i32, vp, i32]),
        "kda_set_debug_checks": (None, [c_int]),
        "kda_debug_checks": (c_int, []),
        "kda_set_test_fault": (c_int, [c_int]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if lib.kda_prefill_args_bytes() != ctypes.sizeof(PrefillArgs):
        raise RuntimeError("kda_prefill_args layout mismatch between include/kda.h and the binding")
    if lib.kda_backward_args_bytes() != ctypes.sizeof(BackwardArgs):
        raise RuntimeError("kda_backward_args layout mismatch between include/kda.h and the binding")
    if lib.kda_fused_decode_args_bytes() != ctypes.sizeof(FusedDecodeArgs):
        raise RuntimeError("kda_fused_decode_args layout mismatch between include/kda.h and the binding")
    _lib = lib
    return lib


# ---------------------------------------------------------------- marshalling helpers

def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("expected contiguous CUDA tensors")


# Shapes and dtypes, checked on the host before the device check and before any call into the library.
# The C ABI takes bare pointers and the kernels trust the extents they are given, so a tensor of the wrong
# shape or dtype would be read or written out of bounds on the device instead of raising here.  A shape
# entry of None accepts any extent.

_FP = (torch.float32,)
_IN = (torch.float32, torch.bfloat16)
_I32 = (torch.int32,)


def _need(name, t, shape, dtypes):
    if t is None:
        return
    if t.dim() != len(shape) or any(s is not None and t.shape[i] != s for i, s in enumerate(shape)):
        want = ", ".join("*" if s is None else str(s) for s in shape)
        raise ValueError(f"{name}: expected shape [{want}], got {list(t.shape)}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: expected dtype {' or '.join(str(d) for d in dtypes)}, got {t.dtype}")


def _need_status(t):
    if t is not None and (t.dtype != torch.int32 or t.numel() < 2):
        raise ValueError(f"dev_status: expected an int32 tensor of at least 2 elements, got {t.dtype} "
                         f"x {t.numel()}")


def _rank(name, t, n):
    if t.dim() != n:
        raise ValueError(f"{name}: expected {n} dimensions, got shape {list(t.shape)}")
    return tuple(t.shape)


def _need_tokens(q, k, v, g, beta, lead):
    """q, k, g [*lead, H, dk]; v [*lead, H, dv] in q's dtype (fp32 or bf16); g fp32; beta [*lead, H] fp32.
    Returns (H, dk, dv)."""
    n = len(lead)
    H, dk = _rank("q", q, n + 2)[n:]
    _need("q", q, (*lead, H, dk), _IN)
    _need("k", k, (*lead, H, dk), (q.dtype,))
    _need("v", v, (*lead, H, None), (q.dtype,))
    dv = v.shape[-1]
    _need("g", g, (*lead, H, dk), _FP)
    _need("beta", beta, (*lead, H), _FP)
    return H, dk, dv


def _need_prefill(q, k, v, g, beta, cu_seqlens, pool, slot_ids, out, extra_pool=None, extra_slot_ids=None):
    T = _rank("q", q, 3)[0]
    H, dk, dv = _need_tokens(q, k, v, g, beta, (T,))
    _need("cu_seqlens", cu_seqlens, (None,), _I32)
    if cu_seqlens.numel() < 1:
        raise ValueError("cu_seqlens: expected N + 1 >= 1 offsets")
    N = cu_seqlens.numel() - 1
    _need("pool", pool, (None, H, dk, dv), _FP)
    _need("slot_ids", slot_ids, (N,), _I32)
    _need("out", out, (T, H, dv), _IN)
    if (extra_pool is None) != (extra_slot_ids is None):
        raise ValueError("extra_pool and extra_slot_ids go together")
    _need("extra_pool", extra_pool, (None, H, dk, dv), _FP)
    _need("extra_slot_ids", extra_slot_ids, (N, 2), _I32)
    return T, N, H, dk, dv


def _need_cfbi_cache(pool, cache, counts):
    S, H = pool.shape[:2]
    _need("cache", cache, (S, H, CFBI_CHUNK, CFBI_ROW_FLOATS), _FP)
    _need("counts", counts, (S, H), _I32)


def _ok(fn: str, code: int):
    if code != KDA_OK:
        raise KdaError(fn, code)


# ---------------------------------------------------------------- entry points

def kda_status_string(code: int) -> str:
    return load().kda_status_string(code).decode()


def kda_version() -> int:
    return load().kda_version()


def kda_check_slot_ids(ids, other_ids=None) -> int:
    """Host-side slot-id contract check on int32 host arrays (numpy or CPU tensors): KDA_OK when the ids are
    distinct and none is among other_ids, else the error code (include/kda.h)."""
    import numpy as np
    a = np.ascontiguousarray(np.asarray(ids), dtype=np.int32)
    b = None if other_ids is None else np.ascontiguousarray(np.asarray(other_ids), dtype=np.int32)
    return load().kda_check_slot_ids(a.ctypes.data if a.size else None, a.size,
                                     None if b is None or not b.size else b.ctypes.data, 0 if b is None else b.size)


def kda_set_debug_checks(on: bool):
    """Switch the library's debug mode (host-side slot-id checks before every call that takes slot ids)."""
    load().kda_set_debug_checks(1 if on else 0)


def kda_set_test_fault(fault: int):
    """Test hook for the kernels' bounded waits (include/kda.h): KDA_TEST_FAULT_STALL_RECORD_INPUTS makes
    kda_prefill_records' first input wait give up and flag KDA_DEV_TIMEOUT; KDA_TEST_FAULT_NONE restores."""
    _ok("kda_set_test_fault", load().kda_set_test_fault(int(fault)))


def kda_debug_checks() -> bool:
    return bool(load().kda_debug_checks())


def kda_state_bytes_per_head(dk: int, dv: int) -> int:
    return load().kda_state_bytes_per_head(dk, dv)


def kda_state_copy(src_pool, src_slots, dst_pool, dst_slots, dev_status=None, stream=None):
    """dst_pool[dst_slots[i]] = src_pool[src_slots[i]] (pools [slots, H, dk, dv] fp32)."""
    head = _rank("src_pool", src_pool, 4)[1:]
    _need("src_pool", src_pool, (None, *head), _FP)
    _need("dst_pool", dst_pool, (None, *head), _FP)
    _need("src_slots", src_slots, (None,), _I32)
    _need("dst_slots", dst_slots, (src_slots.numel(),), _I32)
    _need_status(dev_status)
    _check(src_pool, src_slots, dst_pool, dst_slots, dev_status)
    n = src_slots.numel()
    elems = src_pool[0].numel() if src_pool.shape[0] else dst_pool[0].numel()
    _ok("kda_state_copy", load().kda_state_copy(_p(src_pool), src_pool.shape[0], _p(src_slots), _p(dst_pool),
                                                dst_pool.shape[0], _p(dst_slots), n, elems, _p(dev_status),
                                                _stream(stream)))


def kda_decode_step(q, k, v, g, beta, pool, slot_ids, out, dev_status=None, stream=None):
    """One token per request; q, k, g [B, H, dk]; v, out [B, H, dv]; beta [B, H]; pool updated in place."""
    B = _rank("q", q, 3)[0]
    H, dk, dv = _need_tokens(q, k, v, g, beta, (B,))
    _need("pool", pool, (None, H, dk, dv), _FP)
    _need("slot_ids", slot_ids, (B,), _I32)
    _need("out", out, (B, H, dv), _IN)
    _need_status(dev_status)
    _check(q, k, v, g, beta, pool, slot_ids, out, dev_status)
    B, H, dk = q.shape
    dv = v.shape[-1]
    _ok("kda_decode_step", load().kda_decode_step(_p(q), _p(k), _p(v), _p(g), _p(beta), B, H, dk, dv, _dt(q),
                                                  _p(pool), pool.shape[0], _p(slot_ids), _p(out), _dt(out),
                                                  _p(dev_status), _stream(stream)))


def kda_cfbi_cache_bytes_per_head(dk: int = 128, dv: int = 128) -> int:
    return load().kda_cfbi_cache_bytes_per_head(dk, dv)


def kda_cfbi_prefill(q, k, v, g, beta, cu_seqlens, max_seqlen, pool, cache, counts, slot_ids, out, dev_status=None,
                     stream=None):
    """CF-BI prefill over packed sequences: q, k, g [T, H, 128]; v, out [T, H, 128]; beta [T, H];
    cu_seqlens int32 [N + 1]; pool [S, H, 128, 128]; cache [S, H, 16, 420] fp32; counts [S, H] int32."""
    _need_prefill(q, k, v, g, beta, cu_seqlens, pool, slot_ids, out)
    _need_cfbi_cache(pool, cache, counts)
    _need_status(dev_status)
    _check(q, k, v, g, beta, cu_seqlens, pool, cache, counts, slot_ids, out, dev_status)
    T, H, dk = q.shape
    dv = v.shape[-1]
    N = cu_seqlens.numel() - 1
    _ok("kda_cfbi_prefill", load().kda_cfbi_prefill(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(cu_seqlens), N, T,
                                                    int(max_seqlen), H, dk, dv, _dt(q), _p(pool), _p(cache),
                                                    _p(counts), pool.shape[0], _p(slot_ids), _p(out), _dt(out),
                                                    _p(dev_status), _stream(stream)))


def kda_cfbi_prefill_chunked_workspace_size(T: int, N: int, H: int, dk: int = 128, dv: int = 128) -> int:
    return load().kda_cfbi_prefill_chunked_workspace_size(int(T), int(N), int(H), int(dk), int(dv))


def kda_cfbi_prefill_chunked(q, k, v, g, beta, cu_seqlens, max_seqlen, pool, cache, counts, slot_ids, out,
                             workspace, dev_status=None, stream=None):
    """kda_cfbi_prefill with the chunks worked on in parallel (same arguments and the same bits); workspace is
    a uint8 device tensor of at least kda_cfbi_prefill_chunked_workspace_size(T, N, H) bytes."""
    _need_prefill(q, k, v, g, beta, cu_seqlens, pool, slot_ids, out)
    _need_cfbi_cache(pool, cache, counts)
    _need_status(dev_status)
    _check(q, k, v, g, beta, cu_seqlens, pool, cache, counts, slot_ids, out, dev_status, workspace)
    T, H, dk = q.shape
    dv = v.shape[-1]
    N = cu_seqlens.numel() - 1
    _ok("kda_cfbi_prefill_chunked",
        load().kda_cfbi_prefill_chunked(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(cu_seqlens), N, T, int(max_seqlen),
                                        H, dk, dv, _dt(q), _p(pool), _p(cache), _p(counts), pool.shape[0],
                                        _p(slot_ids), _p(out), _dt(out), _p(workspace),
                                        workspace.numel() * workspace.element_size(), _p(dev_status),
                                        _stream(stream)))


def kda_cfbi_decode(q, k, v, g, beta, pool, cache, counts, slot_ids, out, dev_status=None, stream=None):
    """CF-BI decode, one token per request: q, k, g [B, H, 128]; v, out [B, H, 128]; beta [B, H]."""
    B = _rank("q", q, 3)[0]
    H, dk, dv = _need_tokens(q, k, v, g, beta, (B,))
    _need("pool", pool, (None, H, dk, dv), _FP)
    _need("slot_ids", slot_ids, (B,), _I32)
    _need("out", out, (B, H, dv), _IN)
    _need_cfbi_cache(pool, cache, counts)
    _need_status(dev_status)
    _check(q, k, v, g, beta, pool, cache, counts, slot_ids, out, dev_status)
    B, H, dk = q.shape
    dv = v.shape[-1]
    _ok("kda_cfbi_decode", load().kda_cfbi_decode(_p(q), _p(k), _p(v), _p(g), _p(beta), B, H, dk, dv, _dt(q),
                                                  _p(pool), _p(cache), _p(counts), pool.shape[0], _p(slot_ids),
                                                  _p(out), _dt(out), _p(dev_status), _stream(stream)))


def kda_replay_bytes(B: int, W: int, H: int, dk: int, dv: int, in_dtype: int) -> int:
    return load().kda_replay_bytes(B, W, H, dk, dv, in_dtype)


def kda_verify(q, k, v, g, beta, pool, slot_ids, out, replay, snapshot_out=None, dev_status=None, stream=None):
    """Draft window: q, k, g [B, W, H, dk]; v, out [B, W, H, dv]; beta [B, W, H]; replay: uint8 record buffer."""
    B, W = _rank("q", q, 4)[:2]
    H, dk, dv = _need_tokens(q, k, v, g, beta, (B, W))
    _need("pool", pool, (None, H, dk, dv), _FP)
    _need("slot_ids", slot_ids, (B,), _I32)
    _need("out", out, (B, W, H, dv), _IN)
    _need("snapshot_out", snapshot_out, (B, W, H, dk, dv), _FP)
    _need_status(dev_status)
    _check(q, k, v, g, beta, pool, slot_ids, out, replay, snapshot_out, dev_status)
    B, W, H, dk = q.shape
    dv = v.shape[-1]
    _ok("kda_verify", load().kda_verify(_p(q), _p(k), _p(v), _p(g), _p(beta), B, W, H, dk, dv, _dt(q), _p(pool),
                                        pool.shape[0], _p(slot_ids), _p(out), _dt(out), _p(replay),
                                        replay.numel() * replay.element_size(), _p(snapshot_out), _p(dev_status),
                                        _stream(stream)))


def kda_verify_replay(pool, slot_ids, replay, accepted_len, W, H, dk, dv, in_dtype, dev_status=None, stream=None):
    """Commits tokens 1..accepted_len[b] of each window into pool[slot_ids[b]]."""
    _need("pool", pool, (None, H, dk, dv), _FP)
    _need("slot_ids", slot_ids, (None,), _I32)
    _need("accepted_len", accepted_len, (slot_ids.numel(),), _I32)
    _need_status(dev_status)
    _check(pool, slot_ids, replay, accepted_len, dev_status)
    B = slot_ids.numel()
    _ok("kda_verify_replay", load().kda_verify_replay(_p(pool), pool.shape[0], _p(slot_ids), B, W, H, dk, dv,
                                                      in_dtype, _p(replay), replay.numel() * replay.element_size(),
                                                      _p(accepted_len), _p(dev_status), _stream(stream)))


def _prefill_struct(q, k, v, g, beta, cu_seqlens, max_seqlen, pool, slot_ids, out, init_zero=False,
                    extra_pool=None, extra_slot_ids=None, snapshot_every_chunks=0, workspace=None, dev_status=None):
    _need_prefill(q, k, v, g, beta, cu_seqlens, pool, slot_ids, out, extra_pool, extra_slot_ids)
    _need_status(dev_status)
    _check(q, k, v, g, beta, cu_seqlens, pool, slot_ids, out, extra_pool, extra_slot_ids, workspace, dev_status)
    T, H, dk = q.shape
    a = PrefillArgs()
    a.q, a.k, a.v, a.g, a.beta = (t.data_ptr() for t in (q, k, v, g, beta))
    a.in_dtype = _dt(q)
    a.T, a.H, a.dk, a.dv = T, H, dk, v.shape[-1]
    a.N = cu_seqlens.numel() - 1
    a.cu_seqlens = cu_seqlens.data_ptr()
    a.max_seqlen = int(max_seqlen)
    a.pool, a.num_slots, a.slot_ids = pool.data_ptr(), pool.shape[0], slot_ids.data_ptr()
    a.init_zero = int(bool(init_zero))
    a.out, a.out_dtype = out.data_ptr(), _dt(out)
    if extra_pool is not None:
        a.extra_pool, a.num_extra_slots = extra_pool.data_ptr(), extra_pool.shape[0]
        a.extra_slot_ids = extra_slot_ids.data_ptr()
        a.snapshot_every_chunks = int(snapshot_every_chunks)
    if workspace is not None:
        a.workspace, a.workspace_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    if dev_status is not None:
        a.dev_status = dev_status.data_ptr()
    return a


def kda_prefill_varlen(q, k, v, g, beta, cu_seqlens, max_seqlen, pool, slot_ids, out, init_zero=False,
                       extra_pool=None, extra_slot_ids=None, snapshot_every_chunks=0, workspace=None,
                       dev_status=None, stream=None):
    """Packed prefill: q, k, g [T, H, dk]; v, out [T, H, dv]; beta [T, H]; cu_seqlens int32 [N+1]."""
    a = _prefill_struct(q, k, v, g, beta, cu_seqlens, max_seqlen, pool, slot_ids, out, init_zero, extra_pool,
                        extra_slot_ids, snapshot_every_chunks, workspace, dev_status)
    _ok("kda_prefill_varlen", load().kda_prefill_varlen(ctypes.byref(a), _stream(stream)))


def kda_prefill_records(q, k, v, g, beta, cu_seqlens, max_seqlen, pool, slot_ids, out, init_zero=False,
                        extra_pool=None, extra_slot_ids=None, snapshot_every_chunks=0, workspace=None,
                        dev_status=None, stream=None):
    """Phase 1 of the tensor-core prefill: per-chunk operand records into `workspace`."""
    a = _prefill_struct(q, k, v, g, beta, cu_seqlens, max_seqlen, pool, slot_ids, out, init_zero, extra_pool,
                        extra_slot_ids, snapshot_every_chunks, workspace, dev_status)
    _ok("kda_prefill_records", load().kda_prefill_records(ctypes.byref(a), _stream(stream)))


def kda_prefill_chain(q, k, v, g, beta, cu_seqlens, max_seqlen, pool, slot_ids, out, init_zero=False,
                      extra_pool=None, extra_slot_ids=None, snapshot_every_chunks=0, workspace=None,
                      dev_status=None, stream=None):
    """Phase 2 of the tensor-core prefill: the state carry over the chunks, from the records."""
    a = _prefill_struct(q, k, v, g, beta, cu_seqlens, max_seqlen, pool, slot_ids, out, init_zero, extra_pool,
                        extra_slot_ids, snapshot_every_chunks, workspace, dev_status)
    _ok("kda_prefill_chain", load().kda_prefill_chain(ctypes.byref(a), _stream(stream)))


def kda_prefill_workspace_size(q, k, v, g, beta, cu_seqlens, max_seqlen, pool, slot_ids, out, **kw) -> int:
    a = _prefill_struct(q, k, v, g, beta, cu_seqlens, max_seqlen, pool, slot_ids, out, **kw)
    return load().kda_prefill_workspace_size(ctypes.byref(a))


def kda_segmented_workspace_size(q, k, v, g, beta, cu_seqlens, max_seqlen, pool, slot_ids, out, segment_len,
                                 **kw) -> int:
    a = _prefill_struct(q, k, v, g, beta, cu_seqlens, max_seqlen, pool, slot_ids, out, **kw)
    return load().kda_segmented_workspace_size(ctypes.byref(a), int(segment_len))


def _segmented(fn, q, k, v, g, beta, cu_seqlens, max_seqlen, pool, slot_ids, out, segment_len, workspace,
               init_zero=False, extra_pool=None, extra_slot_ids=None, snapshot_every_chunks=0, dev_status=None,
               stream=None):
    a = _prefill_struct(q, k, v, g, beta, cu_seqlens, max_seqlen, pool, slot_ids, out, init_zero, extra_pool,
                        extra_slot_ids, snapshot_every_chunks, workspace, dev_status)
    _ok(fn, getattr(load(), fn)(ctypes.byref(a), int(segment_len), _stream(stream)))


def kda_prefill_segmented(*args, **kw):
    """Segmented (KCP) prefill; same arguments as kda_prefill_varlen plus segment_len and workspace."""
    _segmented("kda_prefill_segmented", *args, **kw)


def kda_segment_fragments(*args, **kw):
    _segmented("kda_segment_fragments", *args, **kw)


def kda_fragment_scan(*args, **kw):
    _segmented("kda_fragment_scan", *args, **kw)


def kda_segment_outputs(*args, **kw):
    _segmented("kda_segment_outputs", *args, **kw)


def kda_prefill_segmented_noalloc(q, k, v, g, beta, cu_seqlens, max_seqlen, pool, slot_ids, out, segment_len,
                                  init_zero=False, extra_pool=None, extra_slot_ids=None, snapshot_every_chunks=0,
                                  dev_status=None, stream=None):
    """kda_prefill_segmented without a caller workspace: for callers that cannot allocate device memory,
    the scratch comes from a fixed 32 MiB array inside the library (see include/kda.h)."""
    a = _prefill_struct(q, k, v, g, beta, cu_seqlens, max_seqlen, pool, slot_ids, out, init_zero, extra_pool,
                        extra_slot_ids, snapshot_every_chunks, None, dev_status)
    _ok("kda_prefill_segmented_noalloc",
        load().kda_prefill_segmented_noalloc(ctypes.byref(a), int(segment_len), _stream(stream)))


def _backward_struct(q, k, v, g, beta, cu_seqlens, max_seqlen, d_out, dq, dk, dv, dg, dbeta, pool=None,
                     slot_ids=None, d_final=None, d_init=None, workspace=None, dev_status=None):
    T = _rank("q", q, 3)[0]
    H, d_k, d_v = _need_tokens(q, k, v, g, beta, (T,))
    _need("cu_seqlens", cu_seqlens, (None,), _I32)
    if cu_seqlens.numel() < 1:
        raise ValueError("cu_seqlens: expected N + 1 >= 1 offsets")
    N = cu_seqlens.numel() - 1
    if (pool is None) != (slot_ids is None):
        raise ValueError("pool and slot_ids go together (both None: zero initial states)")
    _need("pool", pool, (None, H, d_k, d_v), _FP)
    _need("slot_ids", slot_ids, (N,), _I32)
    _need("d_out", d_out, (T, H, d_v), (q.dtype,))
    for name, t, w in (("dq", dq, d_k), ("dk", dk, d_k), ("dg", dg, d_k), ("dv", dv, d_v)):
        _need(name, t, (T, H, w), _FP)
    _need("dbeta", dbeta, (T, H), _FP)
    _need("d_final", d_final, (N, H, d_k, d_v), _FP)
    _need("d_init", d_init, (N, H, d_k, d_v), _FP)
    _need_status(dev_status)
    _check(q, k, v, g, beta, cu_seqlens, d_out, dq, dk, dv, dg, dbeta, pool, slot_ids, d_final, d_init, workspace,
           dev_status)
    T, H, dkk = q.shape
    a = BackwardArgs()
    a.q, a.k, a.v, a.g, a.beta = (t.data_ptr() for t in (q, k, v, g, beta))
    a.in_dtype = _dt(q)
    a.T, a.H, a.dk, a.dv = T, H, dkk, v.shape[-1]
    a.N = cu_seqlens.numel() - 1
    a.cu_seqlens = cu_seqlens.data_ptr()
    a.max_seqlen = int(max_seqlen)
    if pool is None:
        a.init_zero = 1
    else:
        a.pool, a.num_slots, a.slot_ids = pool.data_ptr(), pool.shape[0], slot_ids.data_ptr()
    a.d_out = d_out.data_ptr()
    a.dq, a.dk_out, a.dv_out, a.dg, a.dbeta = (t.data_ptr() for t in (dq, dk, dv, dg, dbeta))
    if d_final is not None:
        a.d_final = d_final.data_ptr()
    if d_init is not None:
        a.d_init = d_init.data_ptr()
    if workspace is not None:
        a.workspace, a.workspace_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    if dev_status is not None:
        a.dev_status = dev_status.data_ptr()
    return a


def kda_backward_workspace_size(T: int, N: int, H: int, dk: int = 128, dv: int = 128) -> int:
    a = BackwardArgs()
    a.T, a.N, a.H, a.dk, a.dv = T, N, H, dk, dv
    return load().kda_backward_workspace_size(ctypes.byref(a))


def kda_prefill_backward(q, k, v, g, beta, cu_seqlens, max_seqlen, d_out, dq, dk, dv, dg, dbeta, workspace,
                         pool=None, slot_ids=None, d_final=None, d_init=None, dev_status=None, stream=None):
    """Gradients of sum <d_out, o> + <d_final, S_T> through the packed prefill of (q, k, v, g, beta).

    q, k, g, dq, dk, dg [T, H, 128]; v, d_out, dv [T, H, 128]; beta, dbeta [T, H]; cu_seqlens int32 [N + 1];
    initial states pool[slot_ids] (or zero when pool is None); d_final, d_init [N, H, 128, 128] fp32 or None;
    workspace: >= kda_backward_workspace_size(T, N, H) bytes.  Outputs are fp32.
    """
    a = _backward_struct(q, k, v, g, beta, cu_seqlens, max_seqlen, d_out, dq, dk, dv, dg, dbeta, pool, slot_ids,
                         d_final, d_init, workspace, dev_status)
    _ok("kda_prefill_backward", load().kda_prefill_backward(ctypes.byref(a), _stream(stream)))


def kda_fused_decode(xq, xk, xv, a, b, z, pool, slot_ids, conv_state, conv_w, norm_w, out, norm_eps=1e-5,
                     dev_status=None, stream=None):
    """One decode token per request through the short convolution, the KDA step and the gated output norm.

    xq, xk, xv, z, out [B, H, 128]; a [B, H, 128]; b [B, H]; pool [S, H, 128, 128];
    conv_state [S, H, 3, 3, 128] fp32 (advanced in place); conv_w [3, H, 128, 4]; norm_w [128].
    """
    B, H, d = _rank("xq", xq, 3)
    _need("xq", xq, (B, H, d), _IN)
    for name, t in (("xk", xk), ("xv", xv), ("z", z)):
        _need(name, t, (B, H, d), (xq.dtype,))
    _need("a", a, (B, H, d), _FP)
    _need("b", b, (B, H), _FP)
    _need("pool", pool, (None, H, d, d), _FP)
    _need("slot_ids", slot_ids, (B,), _I32)
    _need("conv_state", conv_state, (pool.shape[0], H, 3, 3, d), _FP)
    _need("conv_w", conv_w, (3, H, d, 4), _FP)
    _need("norm_w", norm_w, (d,), _FP)
    _need("out", out, (B, H, d), _IN)
    _need_status(dev_status)
    _check(xq, xk, xv, a, b, z, pool, slot_ids, conv_state, conv_w, norm_w, out, dev_status)
    B, H, d = xq.shape
    f = FusedDecodeArgs()
    f.xq, f.xk, f.xv, f.a, f.b, f.z = (t.data_ptr() for t in (xq, xk, xv, a, b, z))
    f.in_dtype = _dt(xq)
    f.B, f.H, f.dk, f.dv = B, H, d, d
    f.pool, f.num_slots, f.slot_ids = pool.data_ptr(), pool.shape[0], slot_ids.data_ptr()
    f.conv_state, f.conv_w, f.norm_w = conv_state.data_ptr(), conv_w.data_ptr(), norm_w.data_ptr()
    f.norm_eps = float(norm_eps)
    f.out, f.out_dtype = out.data_ptr(), _dt(out)
    if dev_status is not None:
        f.dev_status = dev_status.data_ptr()
    _ok("kda_fused_decode", load().kda_fused_decode(ctypes.byref(f), _stream(stream)))


def kda_kcp_fragments(q, k, v, g, beta, cu_seqlens, max_seqlen, pool, slot_ids, out, segment_len, workspace, frag_out,
                      dev_status=None, stream=None):
    """Fragments (S~ | M) of every segment of the shard's sequences, the last included, into frag_out
    [N, P, H, dk, dv + dk]; run kda_prefill_records on the same workspace first (tensor-core path)."""
    _, N, H, dk, dv = _need_prefill(q, k, v, g, beta, cu_seqlens, pool, slot_ids, out)
    _need("frag_out", frag_out, (N, None, H, dk, dv + dk), _FP)
    _check(frag_out)
    a = _prefill_struct(q, k, v, g, beta, cu_seqlens, max_seqlen, pool, slot_ids, out, workspace=workspace,
                        dev_status=dev_status)
    _ok("kda_kcp_fragments", load().kda_kcp_fragments(ctypes.byref(a), int(segment_len), _p(frag_out),
                                                      _stream(stream)))


def kda_kcp_scan(frags, s0, entries, dev_status=None, stream=None):
    """entries[0] = s0, entries[p + 1] = M_p entries[p] + S~_p over gathered fragments [P, H, dk, dv + dk]."""
    P, H, dk, w = _rank("frags", frags, 4)
    dv = w - dk
    _need("frags", frags, (P, H, dk, dv + dk), _FP)
    _need("s0", s0, (H, dk, dv), _FP)
    _need("entries", entries, (P, H, dk, dv), _FP)
    _need_status(dev_status)
    _check(frags, s0, entries, dev_status)
    P, H, dk, w = frags.shape
    _ok("kda_kcp_scan", load().kda_kcp_scan(_p(frags), P, H, dk, w - dk, _p(s0), _p(entries), _p(dev_status),
                                            _stream(stream)))


def kda_kcp_outputs(q, k, v, g, beta, cu_seqlens, max_seqlen, pool, slot_ids, out, segment_len, workspace, entries,
                    dev_status=None, stream=None):
    """Outputs and final states of the shard from its entry states [N, P, H, dk, dv]."""
    _, N, H, dk, dv = _need_prefill(q, k, v, g, beta, cu_seqlens, pool, slot_ids, out)
    _need("entries", entries, (N, None, H, dk, dv), _FP)
    _check(entries)
    a = _prefill_struct(q, k, v, g, beta, cu_seqlens, max_seqlen, pool, slot_ids, out, workspace=workspace,
                        dev_status=dev_status)
    _ok("kda_kcp_outputs", load().kda_kcp_outputs(ctypes.byref(a), int(segment_len), _p(entries), _stream(stream)))
