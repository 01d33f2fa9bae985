"""Plant plausible mistakes in the oracle (on the CPU) and show that the pins catch each one.

Every mutant replaces one oracle function for the duration of a test and must
fail at least one pin of ``oracle_checks``.
"""
import numpy as np
import pytest

import oracle.attention as oa
import oracle_checks as oc

_attend = oa.attend
_kv_head_of = oa.kv_head_of
_combine = oa.combine


def attend_no_scale(q, k, v, scale, visible=None):
    return _attend(q, k, v, 1.0, visible)


def attend_wrong_sign(q, k, v, scale, visible=None):
    return _attend(q, k, v, -scale, visible)


def attend_lse_without_max(q, k, v, scale, visible=None):
    o, lse = _attend(q, k, v, scale, visible)
    s = scale * (q @ k.T)
    if visible is not None:
        s = np.where(visible, s, -np.inf)
    return o, lse - s.max(axis=1)


def attend_strict_causal(q, k, v, scale, visible=None):
    # off-by-one: a token does not see itself (row 0 then sees nothing -> use key 0 anyway)
    if visible is not None:
        vis = visible.copy()
        n = min(vis.shape)
        vis[np.arange(n), np.arange(n)] = False
        vis[~vis.any(axis=1), 0] = True
        visible = vis
    return _attend(q, k, v, scale, visible)


def attend_mask_after_exp(q, k, v, scale, visible=None):
    # masked scores are dropped from the numerator but still counted in the sum
    s = scale * (q @ k.T)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1)
    if visible is not None:
        e = np.where(visible, e, 0.0)
    return (e @ v) / l[:, None], m[:, 0] + np.log(l)


def attend_transposed_values(q, k, v, scale, visible=None):
    o, lse = _attend(q, k, v, scale, visible)
    return o[::-1].copy(), lse


def kv_head_modulo(hq, Hq, Hkv):
    return hq % Hkv


def combine_unweighted(parts_o, parts_m, parts_l):
    parts_l = np.asarray(parts_l, dtype=np.float64)
    live = parts_l > 0
    o = np.asarray(parts_o)[live].mean(axis=0)
    M = np.asarray(parts_m)[live].max()
    return o, M + np.log(parts_l[live].sum())


def combine_ignores_max(parts_o, parts_m, parts_l):
    parts_l = np.asarray(parts_l, dtype=np.float64)
    live = parts_l > 0
    w = np.where(live, parts_l, 0.0)
    o = (w[:, None] * np.asarray(parts_o)).sum(axis=0) / w.sum()
    return o, np.asarray(parts_m)[live].max() + np.log(w.sum())


def varlen_positions_from_pack_start(q, k, v, cu_seqlens, scale, causal=True, *, heads=None, seqs=None):
    """Causal positions counted from token 0 of the whole pack instead of each sequence's start."""
    q, k, v = oa.f64(q), oa.f64(k), oa.f64(v)
    cu = [int(x) for x in cu_seqlens.tolist()]
    T, Hq, _ = q.shape
    o = np.full((T, Hq, v.shape[2]), np.nan)
    lse = np.full((Hq, T), np.nan)
    for n in range(len(cu) - 1):
        s0, s1 = cu[n], cu[n + 1]
        if s1 <= s0:
            continue
        rows, keys = np.arange(s0, s1), np.arange(0, s1)
        vis = (keys[None, :] <= rows[:, None]) if causal else None
        for h in range(Hq):
            g = oa.kv_head_of(h, Hq, k.shape[1])
            ob, lb = oa.attend(q[s0:s1, h], k[:s1, g], v[:s1, g], scale, vis)
            o[s0:s1, h], lse[h, s0:s1] = ob, lb
    return o, lse


def varlen_shifted_slice(q, k, v, cu_seqlens, scale, causal=True, *, heads=None, seqs=None):
    """Keys and values taken one token late."""
    q, k, v = oa.f64(q), oa.f64(k), oa.f64(v)
    k = np.concatenate([k[1:], k[:1]])
    v = np.concatenate([v[1:], v[:1]])
    return ORIG_VARLEN(q, k, v, cu_seqlens, scale, causal, heads=heads, seqs=seqs)


ORIG_VARLEN = oa.prefill_varlen
ORIG_PAGED = oa.prefill_paged


def chunked_positions_from_zero(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens, scale, causal=True, *,
                                seqs=None, heads=None):
    """New tokens treated as if they opened the sequence (offset dropped)."""
    q = oa.f64(q)
    cu = [int(x) for x in cu_seqlens_q.tolist()]
    lens = [int(x) for x in seq_lens.tolist()]
    T, Hq, _ = q.shape
    o = np.full((T, Hq, v_cache.shape[3]), np.nan)
    lse = np.full((Hq, T), np.nan)
    for n, L in enumerate(lens):
        s0, s1 = cu[n], cu[n + 1]
        if s1 <= s0:
            continue
        keys = oa.gather_pages(oa._PageView(k_cache), block_table[n].tolist(), L, 16)
        vals = oa.gather_pages(oa._PageView(v_cache), block_table[n].tolist(), L, 16)
        pos = np.arange(s1 - s0)
        vis = np.arange(L)[None, :] <= pos[:, None]
        for h in range(Hq):
            g = oa.kv_head_of(h, Hq, k_cache.shape[2])
            ob, lb = oa.attend(q[s0:s1, h], keys[:, g], vals[:, g], scale, vis)
            o[s0:s1, h], lse[h, s0:s1] = ob, lb
    return o, lse


def chunked_keys_of_chunk_only(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens, scale, causal=True, *,
                               seqs=None, heads=None):
    """Only the chunk's own tokens used as keys (the earlier context dropped)."""
    cu = cu_seqlens_q.tolist()
    ql = [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]
    import torch as _t
    return ORIG_PAGED(q, k_cache, v_cache, block_table, cu_seqlens_q, _t.tensor(ql, dtype=_t.int32), scale, causal,
                      seqs=seqs, heads=heads)

MUTANTS = [
    ("attend", attend_no_scale),
    ("attend", attend_wrong_sign),
    ("attend", attend_lse_without_max),
    ("attend", attend_strict_causal),
    ("attend", attend_mask_after_exp),
    ("attend", attend_transposed_values),
    ("kv_head_of", kv_head_modulo),
    ("combine", combine_unweighted),
    ("combine", combine_ignores_max),
    ("prefill_varlen", varlen_positions_from_pack_start),
    ("prefill_varlen", varlen_shifted_slice),
    ("prefill_paged", chunked_positions_from_zero),
    ("prefill_paged", chunked_keys_of_chunk_only),
]


@pytest.mark.parametrize("name,mutant", MUTANTS, ids=[m.__name__ for _, m in MUTANTS])
def test_some_pin_catches(monkeypatch, name, mutant):
    monkeypatch.setattr(oa, name, mutant)
    caught = []
    for check in oc.ALL_CHECKS:
        if check is oc.check_brute_force_tiny and caught:
            continue                     # slow; only needed if nothing else caught it
        try:
            check()
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(check.__name__)
    assert caught, f"no pin catches mutant {mutant.__name__}"
