"""Pins for the float64 oracle: checks against what the pages and the mathematics fix.

Each ``check_*`` raises AssertionError when the oracle disagrees with an
independent fact: a value the pages print, a closed form, an invariant, a
special case that reduces to a library routine, or a brute-force evaluation in
exact / 40-digit arithmetic.  They call the oracle through its module
attributes so that ``test_oracle_mutants`` can plant a mistake in the oracle
and show that some check catches it.
"""
from __future__ import annotations

import json
import math
import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import scipy.special as sps
import torch

import oracle.attention as oa
from workloads import make_chunked_inputs, make_decode_inputs, make_prefill_inputs, make_varlen_inputs, randn_bf16
from workloads.teaching import teaching_scores_values

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _close(a, b, rtol=1e-12, atol=1e-12, what=""):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    err = np.abs(a - b)
    bound = atol + rtol * np.abs(b)
    assert np.all(err <= bound), f"{what}: max err {err.max():.3e}"


# --- values printed by the pages ---------------------------------------------

def check_worked_example_exact():
    """Teaching input of "Plugging in actual numbers": exact output 1.325056137248."""
    g = _golden("worked_example.json")
    s, v = teaching_scores_values(g["tokens"])
    o, _ = oa.attend(np.ones((1, 1)), np.array(s)[:, None], np.array(v)[:, None], 1.0)
    want = float(g["exact_output"])
    assert abs(o[0, 0] - want) < 0.6 * 10.0 ** (-g["exact_output_digits"]), o[0, 0]


def check_worked_example_paged():
    """Same example through the paged decode oracle with shuffled pages (d = 1)."""
    g = _golden("worked_example.json")
    s, v = teaching_scores_values(g["tokens"])
    L = len(s)
    pages = (L + 15) // 16
    perm = np.random.default_rng(7).permutation(pages + 3)[:pages]
    kc = np.full((pages + 3, 16, 1, 1), np.nan)
    vc = np.full((pages + 3, 16, 1, 1), np.nan)
    for p in range(pages):
        n = min(16, L - 16 * p)
        kc[perm[p], :n, 0, 0] = s[16 * p:16 * p + n]
        vc[perm[p], :n, 0, 0] = v[16 * p:16 * p + n]
    o, _ = oa.decode_paged(np.ones((1, 1, 1)), kc, vc, perm[None, :], [L], 1.0)
    assert abs(o[0, 0, 0] - float(g["exact_output"])) < 6e-13, o[0, 0, 0]


# --- closed forms ------------------------------------------------------------

def check_single_key_returns_value():
    """Causal row 0 sees one key: O = v0 exactly, LSE = scale * q0.k0."""
    x = make_prefill_inputs(2, 4, 2, 9, 16, seed=11)
    o, lse = oa.prefill(x.q, x.k, x.v, 0.3, causal=True)
    q, k, v = (oa.f64(t) for t in (x.q, x.k, x.v))
    for b in range(2):
        for h in range(4):
            g = h // 2
            assert np.array_equal(o[b, 0, h], v[b, 0, g]), "row 0 must return v0 exactly"
            exact = float(sum(Fraction(float(a)) * Fraction(float(c)) for a, c in zip(q[b, 0, h], k[b, 0, g])))
            _close(lse[b, h, 0], 0.3 * exact, what="single-key lse")


def check_constant_values():
    """If every visible value is the same vector c, the output is c."""
    x = make_prefill_inputs(1, 2, 1, 33, 8, seed=12)
    c = randn_bf16((1, 1, 1, 8), torch.Generator().manual_seed(3))
    vconst = c.expand(1, 33, 1, 8).contiguous()
    o, _ = oa.prefill(x.q, x.k, vconst, 0.7, causal=True)
    _close(o[0, :, 0, :], np.broadcast_to(oa.f64(c)[0, 0, 0], (33, 8)), rtol=1e-14, what="constant V")


def check_zero_scale_prefix_mean():
    """scale = 0: uniform weights; causal row i is the mean of v[0..i], LSE = ln(i+1)."""
    x = make_prefill_inputs(1, 1, 1, 17, 4, seed=13)
    o, lse = oa.prefill(x.q, x.k, x.v, 0.0, causal=True)
    v = oa.f64(x.v)[0, :, 0, :]
    means = np.cumsum(v, axis=0) / np.arange(1, 18)[:, None]
    _close(o[0, :, 0, :], means, rtol=1e-13, atol=1e-14, what="prefix mean")
    _close(lse[0, 0], np.log(np.arange(1, 18)), what="ln(i+1)")


def check_two_keys_logistic():
    """Two visible keys: weights are the logistic function of the score gap."""
    x = make_prefill_inputs(1, 1, 1, 2, 8, seed=14)
    scale = 0.9
    o, lse = oa.prefill(x.q, x.k, x.v, scale, causal=True)
    q, k, v = (oa.f64(t)[0, :, 0, :] for t in (x.q, x.k, x.v))
    s0, s1 = scale * float(q[1] @ k[0]), scale * float(q[1] @ k[1])
    w1 = sps.expit(s1 - s0)
    _close(o[0, 1, 0], (1 - w1) * v[0] + w1 * v[1], rtol=1e-13, atol=1e-14, what="logistic")
    _close(lse[0, 0, 1], np.logaddexp(s0, s1), what="logaddexp")


def check_noncausal_matches_scipy():
    """Non-causal rows against scipy's softmax / logsumexp routines."""
    x = make_prefill_inputs(1, 2, 2, 23, 16, seed=15)
    o, lse = oa.prefill(x.q, x.k, x.v, 0.25, causal=False)
    q, k, v = (oa.f64(t)[0] for t in (x.q, x.k, x.v))
    for h in range(2):
        s = 0.25 * np.einsum("id,jd->ij", q[:, h], k[:, h])
        _close(o[0, :, h], sps.softmax(s, axis=1) @ v[:, h], rtol=1e-12, atol=1e-13, what="softmax")
        _close(lse[0, h], sps.logsumexp(s, axis=1), what="logsumexp")


# --- invariants -------------------------------------------------------------

def check_weights_sum_to_one():
    """With V = identity the output rows are the weights: >= 0, sum 1, zero above the diagonal."""
    S = 12
    x = make_prefill_inputs(1, 1, 1, S, 8, seed=16)
    eye = torch.eye(S, dtype=torch.float64)[None, :, None, :]
    for causal in (True, False):
        w, _ = oa.prefill(x.q, x.k, eye, 0.5, causal=causal)
        w = w[0, :, 0, :]
        assert np.all(w >= 0)
        _close(w.sum(axis=1), np.ones(S), what="weight sums")
        if causal:
            assert np.all(np.triu(w, 1) == 0.0), "causal weights above the diagonal"
            assert np.all(np.diag(w) > 0.0), "a token must see itself"


def check_max_shift_invariance():
    """Adding c to every score of a row leaves O unchanged and shifts LSE by c."""
    x = make_prefill_inputs(1, 2, 1, 19, 8, seed=17)
    q, k, v = (oa.f64(t) for t in (x.q, x.k, x.v))
    o0, l0 = oa.prefill(q, k, v, 0.5, causal=True)
    for c in (-40.0, 3.0, 250.0):
        q2 = np.concatenate([q, np.ones(q.shape[:3] + (1,))], axis=3)
        k2 = np.concatenate([k, np.full(k.shape[:3] + (1,), c / 0.5)], axis=3)
        o1, l1 = oa.prefill(q2, k2, v, 0.5, causal=True)
        _close(o1, o0, rtol=1e-11, atol=1e-12, what=f"shift {c} output")
        _close(l1, l0 + c, rtol=1e-12, atol=1e-10, what=f"shift {c} lse")


def check_key_permutation_invariance():
    """Non-causal: permuting keys together with their values changes nothing."""
    x = make_prefill_inputs(1, 2, 2, 21, 8, seed=18)
    perm = torch.randperm(21, generator=torch.Generator().manual_seed(4))
    o0, l0 = oa.prefill(x.q, x.k, x.v, 0.4, causal=False)
    o1, l1 = oa.prefill(x.q, x.k[:, perm], x.v[:, perm], 0.4, causal=False)
    _close(o1, o0, rtol=1e-12, atol=1e-13, what="perm output")
    _close(l1, l0, what="perm lse")


def check_causality():
    """Changing keys/values after position i leaves rows <= i bit-identical."""
    x = make_prefill_inputs(1, 2, 1, 16, 8, seed=19)
    o0, l0 = oa.prefill(x.q, x.k, x.v, 0.5, causal=True)
    k2, v2 = x.k.clone(), x.v.clone()
    k2[:, 9:] = -k2[:, 9:] * 3
    v2[:, 9:] = v2[:, 9:] + 5
    o1, l1 = oa.prefill(x.q, k2, v2, 0.5, causal=True)
    assert np.array_equal(o1[:, :9], o0[:, :9]) and np.array_equal(l1[:, :, :9], l0[:, :, :9])
    assert not np.allclose(o1[:, 9:], o0[:, 9:])


def check_gqa_mapping():
    """Query head h reads KV head h // (Hq/Hkv): equals single-head attention on that pair."""
    x = make_prefill_inputs(1, 6, 2, 10, 8, seed=20)
    o, lse = oa.prefill(x.q, x.k, x.v, 0.5, causal=True)
    for h in range(6):
        g = h // 3
        o1, l1 = oa.prefill(x.q[:, :, h:h + 1], x.k[:, :, g:g + 1], x.v[:, :, g:g + 1], 0.5, causal=True)
        assert np.array_equal(o[:, :, h], o1[:, :, 0]) and np.array_equal(lse[:, h], l1[:, 0])


def check_decode_equals_contiguous():
    """Paged decode (shuffled pages, NaN in unused slots) equals attention on the contiguous keys."""
    lens = [1, 15, 16, 17, 40]
    x = make_decode_inputs(lens, Hq=4, Hkv=2, d=8, seed=21, nan_tail=True, extra_blocks=2)
    o, lse = oa.decode_paged(x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens, 0.6)
    kc, vc, q = oa.f64(x.k_cache), oa.f64(x.v_cache), oa.f64(x.q)
    for n, L in enumerate(lens):
        pids = x.block_table[n, :(L + 15) // 16].tolist()
        keys = np.concatenate([kc[p] for p in pids])[:L]
        vals = np.concatenate([vc[p] for p in pids])[:L]
        for h in range(4):
            s = 0.6 * keys[:, h // 2] @ q[n, h]
            w = sps.softmax(s)
            _close(o[n, h], w @ vals[:, h // 2], rtol=1e-12, atol=1e-13, what="decode")
            _close(lse[n, h], sps.logsumexp(s), what="decode lse")
    assert np.isfinite(o).all()


def check_split_combine_invariance():
    """Any split of the keys, merged by the LSE combine, equals the unsplit result."""
    rng = np.random.default_rng(5)
    L, d = 203, 16
    q = rng.standard_normal(d)
    keys = rng.standard_normal((L, d))
    vals = rng.standard_normal((L, d))
    o_ref, l_ref = oa.attend(q[None], keys, vals, 0.8)
    for ns in (1, 2, 4, 16, 7):
        rs = oa.split_ranges(L, num_splits=ns)
        assert rs[0][0] == 0 and rs[-1][1] == L and all(a < b for a, b in rs)
        assert all(rs[i][1] == rs[i + 1][0] for i in range(len(rs) - 1))
        o, lse = oa.decode_split_combine(q, keys, vals, 0.8, rs + [(L, L)])
        _close(o, o_ref[0], rtol=1e-12, atol=1e-13, what=f"{ns} splits")
        _close(lse, l_ref[0], what=f"{ns} splits lse")
    for span in (16, 48, 64, 512):
        rs = oa.split_ranges(L, split_tokens=span)
        o, lse = oa.decode_split_combine(q, keys, vals, 0.8, rs)
        _close(o, o_ref[0], rtol=1e-12, atol=1e-13, what=f"span {span}")


def check_combine_two_groups_closed_form():
    """Two groups: O = (l1 e^m1 o1 + l2 e^m2 o2) / (l1 e^m1 + l2 e^m2); LSE = logaddexp(m1 + ln l1, m2 + ln l2)."""
    o1, o2 = np.array([1.0, -2.0]), np.array([0.5, 4.0])
    m1, m2, l1, l2 = 3.0, -1.5, 2.5, 7.0
    # the middle group is empty (m = -inf, l = 0) and must carry no weight
    o, lse = oa.combine(np.stack([o1, np.zeros(2), o2]), [m1, -np.inf, m2], [l1, 0.0, l2])
    a, b = l1 * math.exp(m1), l2 * math.exp(m2)
    _close(o, (a * o1 + b * o2) / (a + b), rtol=1e-14, what="two-group combine")
    _close(lse, np.logaddexp(m1 + math.log(l1), m2 + math.log(l2)), what="two-group lse")


# --- brute force in exact / 40-digit arithmetic -------------------------------

def _dec_exp(x: Decimal) -> Decimal:
    return x.exp()


def check_brute_force_tiny():
    """Tiny causal problems evaluated with exact dot products and 40-digit exp/ln."""
    getcontext().prec = 40
    for seed, (S, d, Hq, Hkv) in enumerate([(1, 1, 1, 1), (3, 2, 2, 1), (6, 4, 2, 2), (5, 3, 4, 2)]):
        x = make_prefill_inputs(1, Hq, Hkv, S, d, seed=100 + seed)
        scale = 0.375
        o, lse = oa.prefill(x.q, x.k, x.v, scale, causal=True)
        q, k, v = (oa.f64(t)[0] for t in (x.q, x.k, x.v))
        for h in range(Hq):
            g = h // (Hq // Hkv)
            for i in range(S):
                sc = [Decimal(str(float(Fraction(scale) * sum(Fraction(float(q[i, h, t])) * Fraction(float(k[j, g, t]))
                                                              for t in range(d)))))
                      for j in range(i + 1)]
                # the decimal string of a float is exact enough (17 significant digits)
                w = [_dec_exp(s) for s in sc]
                tot = sum(w)
                for t in range(d):
                    num = sum(wj * Decimal(float(v[j, g, t])) for j, wj in enumerate(w))
                    assert abs(float(num / tot) - o[0, i, h, t]) <= 1e-13 * (1 + abs(o[0, i, h, t]))
                assert abs(float(tot.ln()) - lse[0, h, i]) <= 1e-13 * (1 + abs(lse[0, h, i]))


def check_varlen_matches_scipy():
    """Packed sequences: each row against scipy's softmax over its own sequence's keys up to itself."""
    lens = [5, 1, 0, 9, 3]
    x = make_varlen_inputs(lens, Hq=4, Hkv=2, d=6, seed=31, extra=2)
    o, lse = oa.prefill_varlen(x.q, x.k, x.v, x.cu_seqlens, 0.45, causal=True)
    q, k, v = oa.f64(x.q), oa.f64(x.k), oa.f64(x.v)
    cu = x.cu_seqlens.tolist()
    for n in range(len(lens)):
        for i in range(cu[n], cu[n + 1]):
            for h in range(4):
                s = 0.45 * k[cu[n]:i + 1, h // 2] @ q[i, h]
                _close(o[i, h], sps.softmax(s) @ v[cu[n]:i + 1, h // 2], rtol=1e-12, atol=1e-13, what="varlen o")
                _close(lse[h, i], sps.logsumexp(s), what="varlen lse")
    assert np.isnan(o[-2:]).all() and np.isnan(lse[:, -2:]).all()   # tokens in no sequence


def check_varlen_single_token_sequences():
    """A one-token sequence returns its own value row exactly and lse = scale * q.k."""
    x = make_varlen_inputs([1, 1, 1], Hq=2, Hkv=1, d=8, seed=32)
    o, lse = oa.prefill_varlen(x.q, x.k, x.v, x.cu_seqlens, 0.7, causal=False)
    q, k, v = oa.f64(x.q), oa.f64(x.k), oa.f64(x.v)
    for t in range(3):
        for h in range(2):
            assert np.array_equal(o[t, h], v[t, 0])
            _close(lse[h, t], 0.7 * float(q[t, h] @ k[t, 0]), what="single-token lse")


def check_varlen_sequences_isolated():
    """Changing one sequence's tokens leaves every other sequence bit-identical."""
    lens = [7, 4, 6]
    x = make_varlen_inputs(lens, Hq=2, Hkv=2, d=4, seed=33)
    o0, l0 = oa.prefill_varlen(x.q, x.k, x.v, x.cu_seqlens, 0.5, causal=False)
    k2, v2 = x.k.clone(), x.v.clone()
    k2[7:11] = -3 * k2[7:11]
    v2[7:11] = v2[7:11] + 4
    o1, l1 = oa.prefill_varlen(x.q, k2, v2, x.cu_seqlens, 0.5, causal=False)
    keep = np.r_[0:7, 11:17]
    assert np.array_equal(o1[keep], o0[keep]) and np.array_equal(l1[:, keep], l0[:, keep])
    assert not np.allclose(o1[7:11], o0[7:11])


def check_chunked_prefill_matches_scipy():
    """Chunked prefill: each new token against scipy's softmax over the contiguous keys up to its position."""
    ctx, ql = [20, 37, 16, 50, 9], [20, 5, 1, 0, 9]
    x = make_chunked_inputs(ctx, ql, Hq=4, Hkv=2, d=6, seed=34, nan_tail=True, extra_blocks=2)
    o, lse = oa.prefill_paged(x.q, x.k_cache, x.v_cache, x.block_table, x.cu_seqlens_q, x.seq_lens, 0.4)
    q, kc, vc = oa.f64(x.q), oa.f64(x.k_cache), oa.f64(x.v_cache)
    cu = x.cu_seqlens_q.tolist()
    for n, L in enumerate(ctx):
        pids = x.block_table[n, :(L + 15) // 16].tolist()
        keys = np.concatenate([kc[p] for p in pids])[:L]
        vals = np.concatenate([vc[p] for p in pids])[:L]
        for i in range(ql[n]):
            pos = L - ql[n] + i
            for h in range(4):
                s = 0.4 * keys[:pos + 1, h // 2] @ q[cu[n] + i, h]
                _close(o[cu[n] + i, h], sps.softmax(s) @ vals[:pos + 1, h // 2], rtol=1e-12, atol=1e-13,
                       what="chunked o")
                _close(lse[h, cu[n] + i], sps.logsumexp(s), what="chunked lse")


def check_chunked_last_token_is_decode():
    """A one-token chunk at the end of each sequence is exactly the paged decode of that token."""
    ctx = [33, 16, 70]
    x = make_chunked_inputs(ctx, [1, 1, 1], Hq=4, Hkv=1, d=8, seed=35, nan_tail=True)
    o, lse = oa.prefill_paged(x.q, x.k_cache, x.v_cache, x.block_table, x.cu_seqlens_q, x.seq_lens, 0.3)
    od, ld = oa.decode_paged(x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens, 0.3)
    assert np.array_equal(o, od) and np.array_equal(lse, ld.T)


ALL_CHECKS = [
    check_worked_example_exact,
    check_worked_example_paged,
    check_single_key_returns_value,
    check_constant_values,
    check_zero_scale_prefix_mean,
    check_two_keys_logistic,
    check_noncausal_matches_scipy,
    check_weights_sum_to_one,
    check_max_shift_invariance,
    check_key_permutation_invariance,
    check_causality,
    check_gqa_mapping,
    check_decode_equals_contiguous,
    check_split_combine_invariance,
    check_combine_two_groups_closed_form,
    check_varlen_matches_scipy,
    check_varlen_single_token_sequences,
    check_varlen_sequences_isolated,
    check_chunked_prefill_matches_scipy,
    check_chunked_last_token_is_decode,
    check_brute_force_tiny,
]
