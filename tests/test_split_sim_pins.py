"""The scalar split simulation reproduces the numbers the long-context decode page prints.

"Why your local LLM feels dumber than it is" (Part 3.14): sections "Why
FlashAttention 2 selects 54, 62, or 87 groups", "Plugging in actual numbers"
and "GPU specific lowering in Triton".  Values come from tests/golden.
"""
import json
import os

import numpy as np
import pytest

from oracle import numerics as nx
from oracle import split_sim as ss
from workloads.teaching import teaching_scores_values

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")))


@pytest.fixture(scope="module")
def teaching():
    return teaching_scores_values(GOLD["tokens"])


@pytest.mark.parametrize("plat", GOLD["platforms"], ids=lambda p: p["name"])
def test_split_count_heuristic(plat):
    groups, blocks, per = ss.fa2_split_count(GOLD["tokens"], plat["sm_count"])
    assert blocks == GOLD["fa2_blocks"]
    assert groups == plat["groups"]
    assert per == plat["blocks_per_group"]
    assert per * ss.FA2_BLOCK_TOKENS == plat["first_group_tokens"]


@pytest.mark.parametrize("plat", GOLD["platforms"], ids=lambda p: p["name"])
def test_fa2_group_numerics(plat, teaching):
    s, v = teaching
    r = ss.simulate_fa2(s, v, plat["sm_count"])
    assert r.groups == plat["groups"]
    assert r.first_group_tokens == plat["first_group_tokens"]
    assert r.first_local_max == plat["first_local_max"]
    assert f"{r.f32_output:.10f}" == plat["f32_output"]
    assert r.bf16_output == plat["bf16_output"]


def test_exact_reference(teaching):
    s, v = teaching
    assert f"{ss.exact_output(s, v):.12f}" == GOLD["exact_output"]


def test_groups_cover_tokens_once():
    for groups in (1, 7, 54, 62, 87, 431):
        orders = ss.fa2_groups(GOLD["tokens"], groups)
        flat = sorted(t for o in orders for t in o)
        assert flat == list(range(GOLD["tokens"]))


def test_float32_reduction_order():
    tiny = 2.0 ** -24
    left = nx.add(nx.add(1.0, tiny), tiny)
    right = nx.add(1.0, nx.add(tiny, tiny))
    assert float(left) == GOLD["reduction_order"]["left_first"]
    assert repr(float(right)) == GOLD["reduction_order"]["right_first"]


def test_bf16_rounding_neighbours():
    # 1 + 2^-8 is the midpoint between bf16 1.0 and 1.0078125: ties go to even (1.0)
    assert nx.bf16(1.0 + 2.0 ** -8) == 1.0
    assert nx.bf16(1.0 + 3 * 2.0 ** -8) == 1.015625          # midpoint, odd below -> up
    assert nx.bf16(1.0 + 2.0 ** -8 + 2.0 ** -20) == 1.0078125
    assert nx.bf16(-2.5) == -2.5
    assert nx.bf16(1.325056137248) == 1.328125
    assert nx.bf16(1.3241630793) == 1.3203125
    assert np.isnan(nx.bf16(float("nan")))
    arr = nx.bf16_array(np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 3.0], dtype=np.float32))
    assert arr.tolist() == [1.0, 1.015625, 3.0]
