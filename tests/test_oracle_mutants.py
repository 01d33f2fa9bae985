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
