"""Pins for the restated decode-backend numerics (Triton, FlashAttention 2, XQA, TensorRT-LLM).

"Why your local LLM feels dumber than it is" (Part 3.14), section "Backend
names expand into four decode algorithms" fixes each backend's group geometry
and which values it rounds to bfloat16; the page prints numbers only for the
FlashAttention-2 case (pinned in test_split_sim_pins).  The other three are
pinned by what their definitions force:
  * the group counts the page states (XQA: 33 groups on H200, 47 on SM120);
  * every geometry covers each token exactly once, in the stated tile pattern;
  * in exact arithmetic every merge reduces to the plain softmax average
    (a dropped rescale, a wrong weight or a swapped operand breaks this);
  * one group: each merge hands back what that group stored;
  * XQA sums the same bf16 weights it multiplies the values with, so a
    constant power-of-two value comes back exactly; the others do not;
  * shifting every score by an exact constant leaves the max-based merges bit-identical.
Mutants planted in the oracle (on the CPU) show that these pins catch plausible mistakes.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import split_sim as ss
from workloads.teaching import teaching_scores_values

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "decode_backends.json")))
PLATFORMS = (132, 148, 188)


@pytest.fixture(scope="module")
def teaching():
    return teaching_scores_values(GOLD["tokens"])


def _random_case(seed, L):
    rng = np.random.default_rng(seed)
    return list(rng.normal(0.0, 1.5, L)), list(rng.normal(0.0, 1.0, L))


# --- geometry ---------------------------------------------------------------------

def test_geometry_constants_match_the_page():
    assert ss.TRITON_SEGMENTS == GOLD["triton"]["segments"]
    assert ss.TRITON_TILE_TOKENS == GOLD["triton"]["tile_tokens"]
    assert ss.FA2_BLOCK_TOKENS == GOLD["fa2"]["block_tokens"]
    assert ss.XQA_TILE_TOKENS == GOLD["xqa"]["tile_tokens"]
    assert ss.TRT_TILE_TOKENS == GOLD["trt"]["tile_tokens"]


@pytest.mark.parametrize("plat", GOLD["xqa"]["groups"], ids=lambda p: p["name"])
def test_xqa_group_count(plat):
    got = ss.xqa_partition_count(GOLD["tokens"], plat["sm_count"], GOLD["xqa"]["kv_heads"])
    assert got == plat["groups"]


@pytest.mark.parametrize("backend", ss.BACKENDS)
@pytest.mark.parametrize("L", [1, 15, 16, 17, 255, 256, 257, 1000, 27525])
@pytest.mark.parametrize("partitions", [1, 3, 16, 33])
def test_groups_cover_tokens_once(backend, L, partitions):
    groups = ss.backend_groups(backend, L, partitions)
    flat = sorted(t for g in groups for t in g)
    assert flat == list(range(L))
    assert all(g for g in groups)


@pytest.mark.parametrize("L", [1, 300, 4097, 27525])
@pytest.mark.parametrize("partitions", [1, 5, 33])
def test_tile_patterns(L, partitions):
    # XQA: group p holds whole 256-token tiles whose index is p modulo the group count
    for p, g in enumerate(ss.xqa_groups(L, partitions)):
        assert {t // 256 % partitions for t in g} == {p}
        assert all(len([t for t in g if t // 256 == tile]) == min(256, L - 256 * tile) for tile in {t // 256 for t in g})
    # TensorRT-LLM: 128-token tiles in order
    assert [g[0] for g in ss.trt_groups(L)] == list(range(0, L, 128))
    # Triton: at most 16 contiguous groups, all but the last a whole number of 16-token tiles
    tg = ss.triton_groups(L)
    assert len(tg) <= 16 and all(len(g) % 16 == 0 for g in tg[:-1])
    assert all(g == list(range(g[0], g[0] + len(g))) for g in tg)
    # a segment spans ceil(L / 256) tiles (the last one what is left)
    assert len(tg[0]) == min(L, 16 * math.ceil(L / 256))


# --- merges -----------------------------------------------------------------------

@pytest.mark.parametrize("backend", ss.BACKENDS)
@pytest.mark.parametrize("sm", PLATFORMS)
def test_exact_arithmetic_gives_the_softmax_average(backend, sm, teaching):
    s, v = teaching
    got = ss.simulate(backend, s, v, sm, ar=ss.EXACT).f32_output
    assert abs(got - ss.exact_output(s, v)) < 1e-12


@pytest.mark.parametrize("backend", ss.BACKENDS)
@pytest.mark.parametrize("seed,L,partitions", [(1, 700, 3), (2, 4096, 16), (3, 3000, 7), (4, 129, 1)])
def test_exact_merge_identity_random(backend, seed, L, partitions):
    s, v = _random_case(seed, L)
    groups = ss.backend_groups(backend, L, partitions)
    parts = [ss.group_partial(s, v, g, ar=ss.EXACT, **ss.GROUP_OPTIONS[backend]) for g in groups]
    stored = [p.weighted_sum if ss.STORED[backend] == "numerator" else p.normalised_output for p in parts]
    out, lse = ss.merge(backend, stored, [p.local_max for p in parts], [p.norm_sum for p in parts], ss.EXACT)
    top = max(s)
    w = [math.exp(x - top) for x in s]
    assert abs(float(out) - math.fsum(a * b for a, b in zip(w, v)) / math.fsum(w)) < 1e-12
    assert abs(float(lse) - (top + math.log(math.fsum(w)))) < 1e-12


def test_one_group_returns_what_it_stored():
    s, v = _random_case(5, 500)
    g = list(range(500))
    p = ss.group_partial(s, v, g)
    m, l = [p.local_max], [p.norm_sum]
    assert float(ss.merge("triton", [p.weighted_sum], m, l)[0]) == p.normalised_output
    assert float(ss.merge("fa2", [p.normalised_output], m, l)[0]) == p.normalised_output
    want = float(np.float32(ss.FLOAT32.bf16(p.weighted_sum)) / np.float32(p.norm_sum))
    assert float(ss.merge("trt", [p.weighted_sum], m, l)[0]) == want


def test_bf16_weights_in_the_sum_keep_constant_values_exact(teaching):
    s, _ = teaching
    const = [0.5] * len(s)
    # per group: XQA's sum adds exactly the weights its numerator multiplies by 0.5
    for b in ss.BACKENDS:
        groups = ss.backend_groups(b, len(s), 33 if b == "xqa" else 54)
        parts = [ss.group_partial(s, const, g, **ss.GROUP_OPTIONS[b]) for g in groups]
        same = [p.weighted_sum == 0.5 * p.norm_sum for p in parts]
        assert all(same) if b == "xqa" else not any(same), b
    assert ss.simulate("xqa", s, const, 132).f32_output == 0.5
    for b in ("triton", "fa2", "trt"):
        assert ss.simulate(b, s, const, 132).f32_output != 0.5


@pytest.mark.parametrize("backend", ["triton", "xqa", "trt"])
def test_max_based_merges_ignore_an_exact_score_shift(backend, teaching):
    s, v = teaching
    shifted = [x + 3.0 for x in s]  # exact: scores are multiples of 1/8 below 16
    a = ss.simulate(backend, s, v, 132)
    b = ss.simulate(backend, shifted, v, 132)
    assert a.f32_output == b.f32_output


def test_vector_merge_is_the_scalar_merge_per_component():
    rng = np.random.default_rng(9)
    S, d = 6, 5
    part = rng.normal(size=(S, d)).astype(np.float32)
    m = rng.normal(size=S).astype(np.float32)
    l = rng.uniform(1, 50, size=S).astype(np.float32)
    for b in ss.BACKENDS:
        vec, lse = ss.merge(b, part, m, l)
        for x in range(d):
            sc, lse_x = ss.merge(b, part[:, x], m, l)
            assert vec[x] == sc and lse == lse_x


# --- mutants: each plausible mistake must fail a pin above --------------------------

def _triton_unscaled_sum(num, m, l, ar=ss.FLOAT32):
    top = ar.r(max(float(x) for x in m))
    wsum, nsum = ar.r(0.0), ar.r(0.0)
    for i in range(len(m)):
        c = ar.exp(ar.sub(m[i], top))
        wsum = ar.add(wsum, l[i])  # mistake: the sum is not rescaled
        nsum = ar.add(nsum, ar.mul(num[i], c))
    return ar.div(nsum, wsum), ar.add(top, ar.log(wsum))


def _xqa_without_sum_weight(o, m, l, ar=ss.FLOAT32):
    top = ar.r(max(float(x) for x in m))
    wsum, osum = ar.r(0.0), ar.r(0.0)
    for i in range(len(m)):
        w = ar.exp(ar.sub(m[i], top))  # mistake: l_i dropped from the weight
        wsum = ar.add(wsum, w)
        osum = ar.add(osum, ar.mul(o[i], w))
    return ar.div(osum, wsum), ar.add(top, ar.log(wsum))


def _trt_without_running_rescale(num, m, l, ar=ss.FLOAT32):
    run_m, run_l, run_n = -math.inf, ar.r(0.0), ar.r(0.0)
    for i in range(len(m)):
        new_m = max(run_m, float(m[i]))
        take = ar.exp(ar.sub(m[i], new_m))
        run_l = ar.add(run_l, ar.mul(l[i], take))  # mistake: running state kept at its old max
        run_n = ar.add(run_n, ar.mul(ar.bf16(num[i]), take))
        run_m = new_m
    return ar.div(run_n, run_l), ar.add(run_m, ar.log(run_l))


def _fa2_weights_by_max(o, m, l, ar=ss.FLOAT32):
    top = ar.r(max(float(x) for x in m))
    wsum, osum = ar.r(0.0), ar.r(0.0)
    for i in range(len(m)):
        w = ar.exp(ar.sub(m[i], top))  # mistake: max instead of log-sum
        wsum = ar.add(wsum, w)
        osum = ar.add(osum, ar.mul(o[i], w))
    return ar.div(osum, wsum), ar.add(top, ar.log(wsum))


def _xqa_contiguous(tokens, partitions):
    per = math.ceil(tokens / partitions)
    return [list(range(a, min(a + per, tokens))) for a in range(0, tokens, per)]


@pytest.mark.parametrize("backend,mutant", [("triton", _triton_unscaled_sum), ("xqa", _xqa_without_sum_weight),
                                            ("trt", _trt_without_running_rescale), ("fa2", _fa2_weights_by_max)])
def test_mutant_merge_fails_the_identity(backend, mutant, monkeypatch, teaching):
    monkeypatch.setitem(ss.MERGES, backend, mutant)
    with pytest.raises(AssertionError):
        # the teaching input's groups may share one max; the random cases' groups do not
        for sm in PLATFORMS:
            test_exact_arithmetic_gives_the_softmax_average(backend, sm, teaching)
        for seed, L, partitions in [(1, 700, 3), (2, 4096, 16), (3, 3000, 7)]:
            test_exact_merge_identity_random(backend, seed, L, partitions)


def test_mutant_xqa_f32_sum_weights_fails_constant_values(monkeypatch, teaching):
    monkeypatch.setitem(ss.GROUP_OPTIONS, "xqa", {"bf16_output": True})
    with pytest.raises(AssertionError):
        test_bf16_weights_in_the_sum_keep_constant_values_exact(teaching)


def test_mutant_xqa_contiguous_groups_fail_the_tile_pattern(monkeypatch):
    monkeypatch.setattr(ss, "xqa_groups", _xqa_contiguous)
    with pytest.raises(AssertionError):
        test_tile_patterns(4097, 5)


def test_mutant_trt_bf16_weights_in_the_sum_fails_constant_values(monkeypatch, teaching):
    monkeypatch.setitem(ss.GROUP_OPTIONS, "trt", {"bf16_norm_weights": True})
    with pytest.raises(AssertionError):
        test_bf16_weights_in_the_sum_keep_constant_values_exact(teaching)
