"""Exact attention in float64 on the CPU -- test infrastructure, not product code.

Definition: "Why your local LLM feels dumber than it is" (Part 3.14), section
"What attention is trying to calculate".  For one query and the tokens it may
see, score_t = scale * dot(query, key_t); weight_t = exp(score_t) divided by
the sum of exp over the visible tokens; output = sum_t weight_t * value_t.
Subtracting the largest score before exp does not change the result
(section "Why the calculation is split into groups"), so it is done for range.

The log-sum-exp returned beside the output is ln(sum_t exp(score_t)) in
natural-log units, the per-group statistic of that page's simulation.

Readings (the pages leave these open):
  * causal prefill: query i sees keys j <= i (it sees itself);
  * grouped-query attention: query head h reads KV head h // (Hq // Hkv);
  * decode: the single query sees all seq_len cached tokens, gathered through
    the block table (16-token pages);
  * no rounding anywhere: bf16 inputs are widened exactly to float64.
"""
from __future__ import annotations

import math

import numpy as np
import torch


def f64(x) -> np.ndarray:
    """Exact widening of a bf16/f32 tensor (or array) to float64."""
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu").to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def attend(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
           visible: np.ndarray | None = None) -> tuple[np.ndarray, np.ndarray]:
    """Softmax attention of each query row over the keys it may see.

    q [M, d], k [N, d], v [N, dv], visible bool [M, N] (None = all).
    Returns (o [M, dv], lse [M]).  A row that sees no key is an error.
    """
    s = scale * (q @ k.T)
    if visible is not None:
        if not visible.any(axis=1).all():
            raise ValueError("a query row sees no key")
        s = np.where(visible, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)                      # masked entries give exactly 0
    l = e.sum(axis=1)
    o = (e @ v) / l[:, None]
    lse = m[:, 0] + np.log(l)
    return o, lse


def kv_head_of(hq: int, Hq: int, Hkv: int) -> int:
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    return hq // (Hq // Hkv)


def prefill(q, k, v, scale: float, causal: bool = True, *, heads=None, rows=None,
            batches=None) -> tuple[np.ndarray, np.ndarray]:
    """Prefill attention. q [B,S,Hq,d], k/v [B,S,Hkv,d] (torch bf16 or float arrays).

    Returns o [B,S,Hq,d] and lse [B,Hq,S] in float64.  ``heads``/``rows``/
    ``batches`` restrict the work to a sample; entries outside it are NaN.
    """
    q, k, v = f64(q), f64(k), f64(v)
    B, S, Hq, d = q.shape
    Hkv = k.shape[2]
    o = np.full((B, S, Hq, v.shape[3]), np.nan)
    lse = np.full((B, Hq, S), np.nan)
    heads = range(Hq) if heads is None else heads
    batches = range(B) if batches is None else batches
    rows = np.arange(S) if rows is None else np.asarray(rows, dtype=np.int64)
    keys = np.arange(S)
    visible = (keys[None, :] <= rows[:, None]) if causal else None
    for b in batches:
        for hq in heads:
            g = kv_head_of(hq, Hq, Hkv)
            ob, lb = attend(q[b, rows, hq, :], k[b, :, g, :], v[b, :, g, :], scale, visible)
            o[b, rows, hq, :] = ob
            lse[b, hq, rows] = lb
    return o, lse


def prefill_varlen(q, k, v, cu_seqlens, scale: float, causal: bool = True, *, heads=None,
                   seqs=None) -> tuple[np.ndarray, np.ndarray]:
    """Packed sequences, each attended on its own.

    q [T,Hq,d], k/v [T,Hkv,d]; sequence n is tokens cu_seqlens[n] .. cu_seqlens[n+1]-1 and its
    causal positions count from its first token.  Returns o [T,Hq,d] and lse [Hq,T] in float64;
    tokens outside the sampled sequences/heads (or in no sequence) are NaN.  This is the varlen
    attention call of "GPU Datapath: Where Every Byte Moves in One LLM Inference Step", section
    "Measuring the Real Kernels, One at a Time", with the per-row definition of "What attention is
    trying to calculate" ("Why your local LLM feels dumber than it is").
    """
    q, k, v = f64(q), f64(k), f64(v)
    cu = [int(x) for x in (cu_seqlens.tolist() if isinstance(cu_seqlens, torch.Tensor) else cu_seqlens)]
    T, Hq, _ = q.shape
    Hkv = k.shape[1]
    o = np.full((T, Hq, v.shape[2]), np.nan)
    lse = np.full((Hq, T), np.nan)
    heads = range(Hq) if heads is None else heads
    seqs = range(len(cu) - 1) if seqs is None else seqs
    for n in seqs:
        s0, s1 = cu[n], cu[n + 1]
        if s1 <= s0:
            continue
        pos = np.arange(s1 - s0)
        visible = (pos[None, :] <= pos[:, None]) if causal else None
        for hq in heads:
            g = kv_head_of(hq, Hq, Hkv)
            ob, lb = attend(q[s0:s1, hq, :], k[s0:s1, g, :], v[s0:s1, g, :], scale, visible)
            o[s0:s1, hq, :] = ob
            lse[hq, s0:s1] = lb
    return o, lse


class _PageView:
    """Indexing a cache page by page, widening each page to float64 on access."""

    def __init__(self, cache):
        self.cache = cache
        self.shape = tuple(cache.shape)

    def __getitem__(self, p):
        return f64(self.cache[p])


def gather_pages(cache, block_table_row, seq_len: int, page: int) -> np.ndarray:
    """Logical tokens [seq_len, Hkv, d] of one sequence, read through its block table."""
    npages = (seq_len + page - 1) // page
    pids = [int(p) for p in block_table_row[:npages]]
    if npages == 0:
        return np.zeros((0,) + tuple(cache.shape[2:]))
    toks = np.concatenate([cache[p] for p in pids], axis=0)
    return toks[:seq_len]


def decode_paged(q, k_cache, v_cache, block_table, seq_lens, scale: float, *,
                 seqs=None) -> tuple[np.ndarray, np.ndarray]:
    """Single-token decode over a paged cache.

    q [N,Hq,d]; caches [num_blocks, page, Hkv, d]; block_table [N, max_blocks];
    seq_lens [N].  Returns o [N,Hq,d] and lse [N,Hq] in float64.
    """
    q = f64(q)
    bt = np.asarray(block_table.cpu() if isinstance(block_table, torch.Tensor) else block_table)
    lens = [int(x) for x in (seq_lens.tolist() if isinstance(seq_lens, torch.Tensor) else seq_lens)]
    N, Hq, d = q.shape
    page, Hkv, dv = k_cache.shape[1], k_cache.shape[2], v_cache.shape[3]
    o = np.full((N, Hq, dv), np.nan)
    lse = np.full((N, Hq), np.nan)
    for n in (range(N) if seqs is None else seqs):
        if lens[n] == 0:
            continue                     # no key: the result is undefined
        # widen only this sequence's pages (the caches can be large)
        keys = gather_pages(_PageView(k_cache), bt[n], lens[n], page)
        vals = gather_pages(_PageView(v_cache), bt[n], lens[n], page)
        for hq in range(Hq):
            g = kv_head_of(hq, Hq, Hkv)
            on, ln = attend(q[n, hq][None, :], keys[:, g, :], vals[:, g, :], scale)
            o[n, hq] = on[0]
            lse[n, hq] = ln[0]
    return o, lse


# ---------------------------------------------------------------------------
# Split-KV decomposition ("Why the calculation is split into groups"): each
# group of tokens gives a partial (normalised output, local max, local sum);
# the partials are merged with weights l_i * exp(m_i - M).
# ---------------------------------------------------------------------------

def prefill_paged(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens, scale: float, causal: bool = True, *,
                  seqs=None, heads=None) -> tuple[np.ndarray, np.ndarray]:
    """Chunked prefill against a paged cache.

    Sequence n has seq_lens[n] cached tokens (read through its block-table row) and its new tokens
    are q rows cu_seqlens_q[n] .. cu_seqlens_q[n+1]-1, the last ones of the sequence: new token i sits
    at position seq_lens[n] - q_len + i and, causally, sees the keys up to that position.  Returns
    o [T,Hq,d] and lse [Hq,T] in float64 (NaN outside the sampled sequences/heads).  The per-row
    definition is that of "What attention is trying to calculate" ("Why your local LLM feels dumber
    than it is"); the paging follows section D of "GPU Datapath: Where Every Byte Moves in One LLM
    Inference Step".
    """
    q = f64(q)
    bt = np.asarray(block_table.cpu() if isinstance(block_table, torch.Tensor) else block_table)
    cu = [int(x) for x in (cu_seqlens_q.tolist() if isinstance(cu_seqlens_q, torch.Tensor) else cu_seqlens_q)]
    lens = [int(x) for x in (seq_lens.tolist() if isinstance(seq_lens, torch.Tensor) else seq_lens)]
    T, Hq, _ = q.shape
    page, Hkv, dv = k_cache.shape[1], k_cache.shape[2], v_cache.shape[3]
    kc, vc = _PageView(k_cache), _PageView(v_cache)
    o = np.full((T, Hq, dv), np.nan)
    lse = np.full((Hq, T), np.nan)
    heads = range(Hq) if heads is None else heads
    seqs = range(len(lens)) if seqs is None else seqs
    for n in seqs:
        s0, s1, L = cu[n], cu[n + 1], lens[n]
        if s1 <= s0:
            continue
        keys = gather_pages(kc, bt[n], L, page)
        vals = gather_pages(vc, bt[n], L, page)
        pos = L - (s1 - s0) + np.arange(s1 - s0)
        visible = (np.arange(L)[None, :] <= pos[:, None]) if causal else None
        for hq in heads:
            g = kv_head_of(hq, Hq, Hkv)
            ob, lb = attend(q[s0:s1, hq, :], keys[:, g, :], vals[:, g, :], scale, visible)
            o[s0:s1, hq, :] = ob
            lse[hq, s0:s1] = lb
    return o, lse


def split_ranges(seq_len: int, *, num_splits: int = 0, split_tokens: int = 0,
                 page: int = 16) -> list[tuple[int, int]]:
    """Contiguous, page-aligned token ranges of one sequence (empty ranges dropped).

    With ``split_tokens`` > 0 every range has that many tokens (the last one
    fewer); otherwise the pages are shared out as ceil(pages / num_splits)
    pages per range.
    """
    if split_tokens > 0:
        span = split_tokens
    else:
        pages = (seq_len + page - 1) // page
        span = ((pages + num_splits - 1) // num_splits) * page
    return [(a, min(a + span, seq_len)) for a in range(0, seq_len, span)] if span > 0 else []


def partial(q_row: np.ndarray, keys: np.ndarray, vals: np.ndarray, scale: float):
    """One group's partial: (normalised output [dv], local max m, local sum l).

    m is the largest scaled score of the group, l = sum exp(score - m); an empty
    group has m = -inf, l = 0 and output 0.
    """
    if keys.shape[0] == 0:
        return np.zeros(vals.shape[1]), -np.inf, 0.0
    s = scale * (keys @ q_row)
    m = float(s.max())
    e = np.exp(s - m)
    l = float(e.sum())
    return (e @ vals) / l, m, l


def combine(parts_o: np.ndarray, parts_m: np.ndarray, parts_l: np.ndarray):
    """Merge group partials: o [G, dv], m [G], l [G] -> (o [dv], lse).

    Groups with l == 0 (m == -inf) carry no weight.
    """
    parts_m = np.asarray(parts_m, dtype=np.float64)
    parts_l = np.asarray(parts_l, dtype=np.float64)
    live = parts_l > 0
    if not live.any():
        raise ValueError("no group has any token")
    M = parts_m[live].max()
    w = np.where(live, parts_l * np.exp(np.where(live, parts_m, M) - M), 0.0)
    W = w.sum()
    o = (w[:, None] * np.asarray(parts_o, dtype=np.float64)).sum(axis=0) / W
    return o, M + math.log(W)


def decode_split_combine(q_row, keys, vals, scale: float, ranges) -> tuple[np.ndarray, float]:
    """Decode one (sequence, head) by groups and merge; equals ``attend`` exactly in reals."""
    po, pm, pl = [], [], []
    for a, b in ranges:
        o, m, l = partial(q_row, keys[a:b], vals[a:b], scale)
        po.append(o)
        pm.append(m)
        pl.append(l)
    return combine(np.stack(po), np.array(pm), np.array(pl))
