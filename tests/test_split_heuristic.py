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


# ------------------------------------------------------------------ length-aware group size

def _items(lens, Hkv, span_pages):
    return Hkv * sum(-(-(-(-L // 16)) // span_pages) for L in lens)


def test_split_tokens_rule_one_wave(attn):
    """The long-context mix fits one wave of near-equal groups: the smallest such span is chosen."""
    from workloads import LONGCTX, decode_lens_for
    lens = decode_lens_for(LONGCTX)
    max_blocks = max(-(-L // 16) for L in lens)
    for cap in (152, 304, 456, 608):
        t = attn.split_tokens_rule(lens, LONGCTX.Hkv, cap, max_blocks)
        assert t > 0 and t % 16 == 0
        s = t // 16
        assert _items(lens, LONGCTX.Hkv, s) <= cap
        assert s == 32 or _items(lens, LONGCTX.Hkv, s - 1) > cap      # smallest span that fits
        assert 4 * s * cap <= 5 * LONGCTX.Hkv * sum(-(-L // 16) for L in lens)   # near-equal groups
    # the order of the sequences does not matter
    assert attn.split_tokens_rule(lens[::-1], LONGCTX.Hkv, 304, max_blocks) == \
        attn.split_tokens_rule(lens, LONGCTX.Hkv, 304, max_blocks)


def test_split_tokens_rule_several_waves(attn):
    """64 sequences x 8 KV heads need several waves: equal power-of-two groups, about three waves."""
    from workloads import PAGED, decode_lens_for
    lens = decode_lens_for(PAGED)
    max_blocks = max(-(-L // 16) for L in lens)
    work = PAGED.Hkv * sum(-(-L // 16) for L in lens)
    for cap in (304, 456):
        s = attn.split_tokens_rule(lens, PAGED.Hkv, cap, max_blocks) // 16
        assert s >= 32 and s & (s - 1) == 0
        assert s <= max(32, work // (3 * cap)) < 2 * s or s == max_blocks


def test_split_tokens_rule_edges(attn):
    assert attn.split_tokens_rule([0, 0, 0], 2, 304, 10) == 16            # nothing to read
    assert attn.split_tokens_rule([100], 1, 304, 7) == 112                 # one short sequence: one group
    assert attn.split_tokens_rule([122863], 2, 304, 7679) == 16 * 51       # one long one: 2 x 151 groups
    assert attn.split_tokens_rule([10**9], 1, 304, 4) == 64                # clamped to the table's 4 pages
    assert attn.split_tokens_rule([], 1, 304, 4) == 0
    assert attn.split_tokens_rule([5], 0, 304, 4) == 0
    assert attn.split_tokens_rule([5], 1, 0, 4) == 0
    assert attn.split_tokens_rule([5], 1, 304, 0) == 0
