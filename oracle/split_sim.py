"""Scalar simulation of split-KV decode numerics -- test infrastructure.

Restates the arithmetic of the four decode algorithms that "Why your local LLM
feels dumber than it is" (Part 3.14) compares, each with explicit rounding at
every step (section "Backend names expand into four decode algorithms", and
the page's walkthrough program that goes with "Plugging in actual numbers"):

  * Triton: 16 contiguous groups made of whole 16-token tiles; every group
    keeps a float32 weighted-value sum (not normalised), its float32 max and
    its float32 sum of weights; the merge rescales sums and numerators to the
    largest group max.
  * FlashAttention 2: contiguous 64-token blocks, the group count chosen by a
    wave-efficiency rule (section "Why FlashAttention 2 selects 54, 62, or 87
    groups"); every group keeps its float32 normalised output and float32 log
    of its sum; the merge weighs outputs by exp(log-sum - largest log-sum).
  * XQA: 256-token tiles dealt round-robin over a platform-chosen number of
    groups; the bfloat16-rounded weights feed both the numerator and the sum;
    every group rounds its normalised output to bfloat16; the merge weighs it
    by the group's sum rescaled to the largest max.
  * TensorRT-LLM: one group per 128-token tile; the reducer takes the
    bfloat16-rounded weighted-value sum with float32 max and sum, and merges
    the groups one after another with a running max.

Inside every group (section "Why the calculation is split into groups") the
exponentials are taken against the group's own max, and the weighted-value sum
uses the weights rounded to bfloat16; only XQA also rounds the weights that
enter the sum.  The simulation works on already-scaled scores and one scalar
value per token, as the page's worked example does; its merges also take
arrays of partial outputs (one float32 row per group), which is how the tests
check the GPU merge kernel element by element.  An ``Arithmetic`` object
decides the rounding: ``FLOAT32`` rounds every result to float32 (bfloat16
where a step says so); ``EXACT`` rounds nothing (float64), in which every merge
must give the plain softmax average -- the identity the tests pin.

The exact float64 attention lives in ``oracle.attention``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from . import numerics as nx

FA2_BLOCK_TOKENS = 64
TRITON_SEGMENTS = 16
TRITON_TILE_TOKENS = 16
XQA_TILE_TOKENS = 256
TRT_TILE_TOKENS = 128
BACKENDS = ("triton", "fa2", "xqa", "trt")


# --- arithmetic models --------------------------------------------------------

class Arithmetic:
    """Rounding model: results of add / sub / mul / div / exp / log are rounded to
    ``dtype``; ``bf16`` is the extra rounding a step may ask for."""

    def __init__(self, name: str, dtype, to_bf16):
        self.name, self.dtype, self._to_bf16 = name, dtype, to_bf16

    def r(self, x) -> np.ndarray:
        return np.asarray(x, dtype=self.dtype)

    def add(self, a, b):
        return self.r(self.r(a) + self.r(b))

    def sub(self, a, b):
        return self.r(self.r(a) - self.r(b))

    def mul(self, a, b):
        return self.r(self.r(a) * self.r(b))

    def div(self, a, b):
        return self.r(self.r(a) / self.r(b))

    def exp(self, x):
        """exp of a scalar, evaluated in double and rounded once."""
        return self.r(math.exp(float(x)))

    def log(self, x):
        return self.r(math.log(float(x)))

    def bf16(self, x):
        return self._to_bf16(self.r(x))


FLOAT32 = Arithmetic("float32", np.float32, nx.bf16_array)
EXACT = Arithmetic("exact", np.float64, lambda x: np.asarray(x, dtype=np.float64))


# --- group geometries ---------------------------------------------------------

def _runs(tokens: int, starts, width: int) -> list[int]:
    out = []
    for a in starts:
        out.extend(range(a, min(a + width, tokens)))
    return out


def triton_groups(tokens: int, segments: int = TRITON_SEGMENTS) -> list[list[int]]:
    """``segments`` contiguous groups, each ceil(tokens / (segments * 16)) 16-token tiles long."""
    span = TRITON_TILE_TOKENS * math.ceil(tokens / (segments * TRITON_TILE_TOKENS))
    return [list(range(a, min(a + span, tokens))) for a in range(0, tokens, span)] if span else []


def fa2_split_count(tokens: int, sm_count: int, kv_heads: int = 4,
                    max_splits: int = 128) -> tuple[int, int, int]:
    """Group count chosen by the wave-efficiency heuristic.

    Capacity is two work blocks per SM.  A candidate group count c is kept
    only if it changes the number of 64-token blocks per group compared with
    c - 1.  Its efficiency is w / ceil(w) with w = kv_heads * c / capacity.
    The smallest kept c whose efficiency is at least 85% of the best wins.
    Returns (groups, total 64-token blocks, blocks per group).
    """
    blocks = math.ceil(tokens / FA2_BLOCK_TOKENS)
    capacity = 2 * sm_count
    limit = min(max_splits, capacity, blocks)
    kept = []
    for c in range(1, limit + 1):
        if c > 1 and math.ceil(blocks / c) == math.ceil(blocks / (c - 1)):
            continue
        waves = kv_heads * c / capacity
        kept.append((c, waves / math.ceil(waves)))
    best = max(eff for _, eff in kept)
    chosen = min(c for c, eff in kept if eff >= 0.85 * best)
    return chosen, blocks, math.ceil(blocks / chosen)


def fa2_groups(tokens: int, groups: int) -> list[list[int]]:
    """Token visiting order of each group: contiguous 64-token blocks, last block first."""
    blocks = math.ceil(tokens / FA2_BLOCK_TOKENS)
    per = math.ceil(blocks / groups)
    out = []
    for gi in range(groups):
        first, stop = gi * per, min(gi * per + per, blocks)
        order = _runs(tokens, [b * FA2_BLOCK_TOKENS for b in reversed(range(first, stop))], FA2_BLOCK_TOKENS)
        if order:
            out.append(order)
    return out


def xqa_partition_count(tokens: int, sm_count: int, kv_heads: int = 4, batch: int = 1) -> int:
    """SMs shared out over (sequence, KV head) pairs, but no more groups than 256-token tiles."""
    return min(max(1, sm_count // (batch * kv_heads)), math.ceil(tokens / XQA_TILE_TOKENS))


def xqa_groups(tokens: int, partitions: int) -> list[list[int]]:
    """Group p takes the 256-token tiles p, p + partitions, p + 2 partitions, ..."""
    tiles = math.ceil(tokens / XQA_TILE_TOKENS)
    out = []
    for p in range(partitions):
        order = _runs(tokens, [t * XQA_TILE_TOKENS for t in range(p, tiles, partitions)], XQA_TILE_TOKENS)
        if order:
            out.append(order)
    return out


def trt_groups(tokens: int) -> list[list[int]]:
    """One group per 128-token tile."""
    return [list(range(a, min(a + TRT_TILE_TOKENS, tokens))) for a in range(0, tokens, TRT_TILE_TOKENS)]


def backend_groups(backend: str, tokens: int, partitions: int = 0) -> list[list[int]]:
    """Groups of one sequence of ``tokens`` tokens; ``partitions`` is the group count where
    the backend takes one (Triton segments, FlashAttention-2 groups, XQA groups)."""
    if backend == "triton":
        return triton_groups(tokens, partitions or TRITON_SEGMENTS)
    if backend == "fa2":
        return fa2_groups(tokens, partitions)
    if backend == "xqa":
        return xqa_groups(tokens, partitions)
    if backend == "trt":
        return trt_groups(tokens)
    raise ValueError(backend)


# --- one group ----------------------------------------------------------------

@dataclass
class GroupState:
    tokens: int
    local_max: float
    norm_sum: float
    weighted_sum: float
    normalised_output: float
    log_sum: float


def group_partial(scores, values, order, *, bf16_norm_weights: bool = False, bf16_output: bool = False,
                  ar: Arithmetic = FLOAT32) -> GroupState:
    """One group: exponentials against the group max, bf16 weights in the numerator.

    ``bf16_norm_weights``: the sum of weights also adds the bf16-rounded weights (XQA).
    ``bf16_output``: the normalised output is rounded to bf16 (XQA).
    """
    m = ar.r(max(scores[t] for t in order))
    l = ar.r(0.0)
    acc = ar.r(0.0)
    for t in order:
        e = ar.exp(ar.r(float(scores[t]) - float(m)))  # the score itself is not rounded first
        eb = ar.bf16(e)
        l = ar.add(l, eb if bf16_norm_weights else e)
        acc = ar.add(acc, ar.mul(eb, ar.bf16(values[t])))
    o = ar.div(acc, l)
    if bf16_output:
        o = ar.bf16(o)
    lse = ar.add(m, ar.log(l))
    return GroupState(len(order), float(m), float(l), float(acc), float(o), float(lse))


# --- merges -------------------------------------------------------------------
# Each takes the groups in order: part [S] or [S, d] (the group's stored output),
# m [S] (group max), l [S] (group sum of weights); no group may be empty.  Each
# returns (output, lse), where lse = log of the merged sum of exp(score), which
# the page does not print: it is the largest max (or log-sum) plus the log of the
# merged sum, rounded like every other step.

def merge_f32_numerators(num, m, l, ar: Arithmetic = FLOAT32):
    """Triton: rescale numerators and sums to the largest max, add in group order, divide."""
    top = ar.r(max(float(x) for x in m))
    wsum, nsum = ar.r(0.0), ar.r(0.0)
    for i in range(len(m)):
        c = ar.exp(ar.sub(m[i], top))
        wsum = ar.add(wsum, ar.mul(l[i], c))
        nsum = ar.add(nsum, ar.mul(num[i], c))
    return ar.div(nsum, wsum), ar.add(top, ar.log(wsum))


def merge_by_log_sums(o, m, l, ar: Arithmetic = FLOAT32):
    """FlashAttention 2: weights exp(lse_i - largest lse) on normalised outputs, lse_i = m_i + log l_i."""
    lse = [ar.add(m[i], ar.log(l[i])) for i in range(len(m))]
    top = ar.r(max(float(x) for x in lse))
    wsum, osum = ar.r(0.0), ar.r(0.0)
    for i in range(len(m)):
        w = ar.exp(ar.sub(lse[i], top))
        wsum = ar.add(wsum, w)
        osum = ar.add(osum, ar.mul(o[i], w))
    return ar.div(osum, wsum), ar.add(top, ar.log(wsum))


def merge_bf16_normalised(o, m, l, ar: Arithmetic = FLOAT32):
    """XQA: a group's (bf16) normalised output weighs l_i exp(m_i - largest max)."""
    top = ar.r(max(float(x) for x in m))
    wsum, osum = ar.r(0.0), ar.r(0.0)
    for i in range(len(m)):
        w = ar.mul(l[i], ar.exp(ar.sub(m[i], top)))
        wsum = ar.add(wsum, w)
        osum = ar.add(osum, ar.mul(o[i], w))
    return ar.div(osum, wsum), ar.add(top, ar.log(wsum))


def merge_ordered_bf16_numerators(num, m, l, ar: Arithmetic = FLOAT32):
    """TensorRT-LLM reducer: one group after another, a running max rescales the running state
    (by 0 before the first group) and the new group's sum and bf16-rounded numerator."""
    run_m = -math.inf
    run_l, run_n = ar.r(0.0), ar.r(0.0)
    for i in range(len(m)):
        new_m = max(run_m, float(m[i]))
        keep = ar.r(0.0) if run_m == -math.inf else ar.exp(ar.sub(run_m, new_m))
        take = ar.exp(ar.sub(m[i], new_m))
        run_l = ar.add(ar.mul(run_l, keep), ar.mul(l[i], take))
        run_n = ar.add(ar.mul(run_n, keep), ar.mul(ar.bf16(num[i]), take))
        run_m = new_m
    return ar.div(run_n, run_l), ar.add(run_m, ar.log(run_l))


MERGES = {
    "triton": merge_f32_numerators,
    "fa2": merge_by_log_sums,
    "xqa": merge_bf16_normalised,
    "trt": merge_ordered_bf16_numerators,
}

# Which stored value each backend's merge takes: the group's weighted-value sum ("numerator")
# or its normalised output; XQA's groups round both their weights-sum inputs and output to bf16.
STORED = {"triton": "numerator", "fa2": "normalised", "xqa": "normalised", "trt": "numerator"}
GROUP_OPTIONS = {
    "triton": {},
    "fa2": {},
    "xqa": {"bf16_norm_weights": True, "bf16_output": True},
    "trt": {},
}


def merge(backend: str, part, m, l, ar: Arithmetic = FLOAT32):
    return MERGES[backend](part, m, l, ar)


# --- whole simulations ----------------------------------------------------------

@dataclass
class SplitResult:
    groups: int
    first_group_tokens: int
    first_local_max: float
    f32_output: float
    bf16_output: float


def simulate(backend: str, scores, values, sm_count: int, kv_heads: int = 4,
             ar: Arithmetic = FLOAT32) -> SplitResult:
    """One backend on scalar scores and values, with the group count the platform implies."""
    L = len(scores)
    if backend == "fa2":
        partitions = fa2_split_count(L, sm_count, kv_heads)[0]
    elif backend == "xqa":
        partitions = xqa_partition_count(L, sm_count, kv_heads)
    else:
        partitions = TRITON_SEGMENTS
    orders = backend_groups(backend, L, partitions)
    parts = [group_partial(scores, values, o, ar=ar, **GROUP_OPTIONS[backend]) for o in orders]
    stored = [p.weighted_sum if STORED[backend] == "numerator" else p.normalised_output for p in parts]
    out, _ = merge(backend, stored, [p.local_max for p in parts], [p.norm_sum for p in parts], ar)
    return SplitResult(len(parts), parts[0].tokens, parts[0].local_max, float(out), float(ar.bf16(out)))


def simulate_fa2(scores, values, sm_count: int, kv_heads: int = 4) -> SplitResult:
    return simulate("fa2", scores, values, sm_count, kv_heads)


def exact_output(scores, values) -> float:
    """Real-number softmax average with exactly rounded sums (math.fsum)."""
    top = max(scores)
    w = [math.exp(s - top) for s in scores]
    return math.fsum(a * b for a, b in zip(w, values)) / math.fsum(w)
