"""Scalar simulation of split-KV decode numerics -- test infrastructure.

Restates, in float32/bfloat16 arithmetic, the FlashAttention-2-like group split
of "Why your local LLM feels dumber than it is" (Part 3.14):

  * section "Why FlashAttention 2 selects 54, 62, or 87 groups": the number of
    groups is chosen by a wave-efficiency heuristic over 64-token blocks;
  * section "Why the calculation is split into groups": inside a group the
    exponentials are taken against the group's own maximum; the weighted-value
    sum uses the weights rounded to bfloat16, the normalisation sum uses the
    unrounded float32 weights;
  * section "Backend names expand into four decode algorithms": the groups
    are contiguous runs of 64-token blocks (visited from the last block of a
    group back to its first), each stores a float32 normalised output and a
    float32 log-sum, and the merge weighs group outputs by exp(lse_i - max lse).

It works on already-scaled scores and one scalar value per token, as the page's
worked example does ("Plugging in actual numbers").  Its role is to pin the
reading of the split and merge arithmetic against the numbers the page prints;
the exact float64 definition lives in ``oracle.attention``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

from . import numerics as nx

FA2_BLOCK_TOKENS = 64


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
        order = []
        for blk in reversed(range(first, stop)):
            order.extend(range(blk * FA2_BLOCK_TOKENS, min((blk + 1) * FA2_BLOCK_TOKENS, tokens)))
        if order:
            out.append(order)
    return out


@dataclass
class GroupState:
    tokens: int
    local_max: float
    norm_sum: float
    weighted_sum: float
    normalised_output: float
    log_sum: float


def group_partial(scores, values, order) -> GroupState:
    """One group in float32: bf16-rounded weights in the numerator, f32 weights in the sum."""
    m = nx.f32(max(scores[t] for t in order))
    l = nx.f32(0.0)
    acc = nx.f32(0.0)
    for t in order:
        e = nx.exp32(nx.f32(float(scores[t]) - float(m)))
        l = nx.add(l, e)
        acc = nx.add(acc, nx.mul(nx.bf16(e), nx.bf16(values[t])))
    o = nx.div(acc, l)
    lse = nx.add(m, nx.log32(l))
    return GroupState(len(order), float(m), float(l), float(acc), float(o), float(lse))


def merge_by_log_sums(parts: list[GroupState]) -> float:
    """Weights exp(lse_i - max lse) in float32, accumulated in group order."""
    top = nx.f32(max(p.log_sum for p in parts))
    wsum = nx.f32(0.0)
    osum = nx.f32(0.0)
    for p in parts:
        w = nx.exp32(nx.f32(p.log_sum - float(top)))
        wsum = nx.add(wsum, w)
        osum = nx.add(osum, nx.mul(p.normalised_output, w))
    return float(nx.div(osum, wsum))


@dataclass
class SplitResult:
    groups: int
    first_group_tokens: int
    first_local_max: float
    f32_output: float
    bf16_output: float


def simulate_fa2(scores, values, sm_count: int, kv_heads: int = 4) -> SplitResult:
    groups, _, _ = fa2_split_count(len(scores), sm_count, kv_heads)
    orders = fa2_groups(len(scores), groups)
    parts = [group_partial(scores, values, o) for o in orders]
    out = merge_by_log_sums(parts)
    return SplitResult(len(parts), parts[0].tokens, parts[0].local_max, out, float(nx.bf16(out)))


def exact_output(scores, values) -> float:
    """Real-number softmax average with exactly rounded sums (math.fsum)."""
    top = max(scores)
    w = [math.exp(s - top) for s in scores]
    return math.fsum(a * b for a, b in zip(w, values)) / math.fsum(w)
