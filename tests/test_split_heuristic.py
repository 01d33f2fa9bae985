"""The C split-count rule against the oracle's restatement and the page's worked numbers (no GPU).

"Why your local LLM feels dumber than it is" (Part 3.14), section "Why FlashAttention 2 selects
54, 62, or 87 groups": 27,525 tokens in 64-token blocks (431), four KV heads, capacity twice the
SM count, 85% of the best estimated efficiency.
"""
import math

import numpy as np
import pytest

import oracle.split_sim as ss


@pytest.mark.parametrize("sms,want", [(132, 54), (148, 62), (188, 87)])
def test_page_platforms(attn, sms, want):
    blocks = math.ceil(27525 / 64)
    assert blocks == 431
    assert attn.split_heuristic(4, 2 * sms, blocks, 128) == want


def test_matches_oracle_rule(attn):
    rng = np.random.default_rng(7)
    for _ in range(3000):
        tokens = int(rng.integers(1, 200_000))
        sms = int(rng.integers(1, 400))
        heads = int(rng.integers(1, 64))
        max_splits = int(rng.integers(1, 200))
        want, blocks, _ = ss.fa2_split_count(tokens, sms, kv_heads=heads, max_splits=max_splits)
        got = attn.split_heuristic(heads, 2 * sms, blocks, max_splits)
        assert got == want, (tokens, sms, heads, max_splits)


def test_invalid_arguments(attn):
    assert attn.split_heuristic(0, 10, 10, 10) == 0
    assert attn.split_heuristic(4, 0, 10, 10) == 0
    assert attn.split_heuristic(4, 10, 0, 10) == 0
    assert attn.split_heuristic(4, 10, 10, 0) == 0
    assert attn.lib().attn_decode_auto_splits(0, 8, 128, 10) == 0
    assert attn.lib().attn_decode_auto_splits(4, 8, 96, 10) == 0


def test_single_block_never_splits(attn):
    assert attn.split_heuristic(1, 296, 1, 128) == 1
