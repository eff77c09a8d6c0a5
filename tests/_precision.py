"""Rounding of fp64 values to the tensor-core operand formats, and products with split operands (numpy;
test helpers for the operand-precision budgets).  bf16: round to nearest even of the fp32 value; tf32: the
fp32 value with its 13 low mantissa bits dropped (truncated) or rounded to nearest (ties away)."""
from __future__ import annotations

import numpy as np


def _bits(x):
    return np.asarray(x, np.float64).astype(np.float32).view(np.uint32)


def _back(b):
    return b.view(np.float32).astype(np.float64)


def f32(x):
    return np.asarray(x, np.float64).astype(np.float32).astype(np.float64)


def bf16(x):
    b = _bits(x)
    b = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return _back(b & np.uint32(0xFFFF0000))


def tf32_trunc(x):
    return _back(_bits(x) & np.uint32(0xFFFFE000))


def tf32_round(x):
    return _back((_bits(x) + np.uint32(0x1000)) & np.uint32(0xFFFFE000))


def split(x):
    """bf16 hi and lo parts: hi = bf16(x), lo = bf16(x - hi)."""
    hi = bf16(x)
    return hi, bf16(x - hi)


def product(a, b, fa, fb):
    """a @ b with each operand exact ("exact"), in single bf16 ("bf16") or split into bf16 hi + lo
    ("split"; the three-term product hi*hi + lo*hi + hi*lo)."""
    def parts(x, fmt):
        if fmt == "exact":
            return x, None
        if fmt == "bf16":
            return bf16(x), None
        return split(x)
    ah, al = parts(a, fa)
    bh, bl = parts(b, fb)
    r = ah @ bh
    if al is not None:
        r = r + al @ bh
    if bl is not None:
        r = r + ah @ bl
    return r
