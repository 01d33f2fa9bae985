"""Float32 and bfloat16 rounding helpers -- test infrastructure.

"Why your local LLM feels dumber than it is" (Part 3.14) models the GPU's
arithmetic with explicit rounding: every float32 operation is rounded to the
nearest float32 (ties to even), and a float32 is rounded to bfloat16 by keeping
its top 16 bits with round-to-nearest-even on the dropped half.  These helpers
implement those two roundings with numpy; they are pinned by tests against the
page's float32 reduction-order example and against known bfloat16 neighbours.
"""
from __future__ import annotations

import math

import numpy as np


def f32(x) -> np.float32:
    """Round a real (python float / float64) to the nearest float32."""
    return np.float32(x)


def bf16(x) -> np.float32:
    """Round to float32, then to bfloat16 (nearest, ties to even); returned as float32."""
    a = np.asarray(np.float32(x), dtype=np.float32)
    bits = a.view(np.uint32).astype(np.uint64)
    if np.isnan(a):
        return np.float32(a)
    lsb = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + lsb) & 0xFFFF0000).astype(np.uint32)
    return rounded.view(np.float32)[()]


def bf16_array(x: np.ndarray) -> np.ndarray:
    """Vectorised ``bf16`` for float32 arrays (NaN passes through)."""
    a = np.asarray(x, dtype=np.float32)
    bits = a.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    out = ((bits + 0x7FFF + lsb) & 0xFFFF0000).astype(np.uint32).view(np.float32)
    return np.where(np.isnan(a), a, out)


def add(a, b) -> np.float32:
    return np.float32(np.float32(a) + np.float32(b))


def mul(a, b) -> np.float32:
    return np.float32(np.float32(a) * np.float32(b))


def div(a, b) -> np.float32:
    return np.float32(np.float32(a) / np.float32(b))


def exp32(x) -> np.float32:
    """exp evaluated in double precision and rounded once to float32."""
    return np.float32(math.exp(float(x)))


def log32(x) -> np.float32:
    return np.float32(math.log(float(x)))
