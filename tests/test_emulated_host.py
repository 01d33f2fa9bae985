"""Host side of the emulated decode numerics (no GPU): group counts, slots and argument checks.

"Why your local LLM feels dumber than it is" (Part 3.14), section "Backend names expand into four
decode algorithms": Triton always uses 16 groups, FlashAttention 2 the 54 / 62 / 87 of its
split rule, XQA 33 groups on H200 and 47 on SM120, TensorRT-LLM one group per 128-token tile.
The C arithmetic is checked against the oracle's restatement and the page's numbers.
"""
import ctypes
import json
import math
import os

import numpy as np
import pytest

import oracle.split_sim as ss

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "decode_backends.json")))
FAKE = 1 << 20


@pytest.mark.parametrize("sm,fa2,xqa", [(132, 54, 33), (148, 62, 37), (188, 87, 47)])
def test_page_group_counts(attn, sm, fa2, xqa):
    L = GOLD["tokens"]
    assert attn.emulated_partitions("triton", 1, 4, L, sm) == GOLD["triton"]["segments"]
    assert attn.emulated_partitions("fa2", 1, 4, L, sm) == fa2
    assert attn.emulated_partitions("xqa", 1, 4, L, sm) == xqa
    assert attn.emulated_partitions("trt", 1, 4, L, sm) == math.ceil(L / GOLD["trt"]["tile_tokens"])


def test_xqa_counts_stated_by_the_page(attn):
    for plat in GOLD["xqa"]["groups"]:
        assert attn.emulated_partitions("xqa", 1, GOLD["xqa"]["kv_heads"], GOLD["tokens"],
                                        plat["sm_count"]) == plat["groups"]


def test_counts_match_the_oracle(attn):
    rng = np.random.default_rng(11)
    for _ in range(2000):
        L = int(rng.integers(1, 300_000))
        sm = int(rng.integers(1, 400))
        heads = int(rng.integers(1, 16))
        assert attn.emulated_partitions("fa2", 1, heads, L, sm) == ss.fa2_split_count(L, sm, heads)[0]
        assert attn.emulated_partitions("xqa", 1, heads, L, sm) == ss.xqa_partition_count(L, sm, heads)
        assert attn.emulated_partitions("trt", 1, heads, L, sm) == len(ss.trt_groups(L))
        assert attn.emulated_partitions("xqa", 2, heads, L, sm) == ss.xqa_partition_count(L, sm, heads, batch=2)


def test_slots_and_workspace(attn):
    assert attn.emulated_num_slots("trt", 1721) == 216        # 27,525 tokens in 16-token pages
    assert attn.emulated_num_slots("trt", 8) == 1
    assert attn.emulated_num_slots("trt", 9) == 2
    for name in ("triton", "fa2", "xqa"):
        assert attn.emulated_num_slots(name, 100, 33) == 33
        assert attn.emulated_num_slots(name, 100, 0) == 0
    assert attn.emulated_num_slots("fa2", 100, 16, page_size=32) == 0
    lib = attn.lib()
    assert lib.attn_emulated_workspace_bytes(2, 8, 128, 1) == 2 * 8 * 1 * 130 * 4
    assert lib.attn_emulated_workspace_bytes(0, 8, 128, 1) == 0
    assert lib.attn_emulated_partitions(5, 1, 4, 100, 132) == 0
    assert lib.attn_emulated_partitions(1, 0, 4, 100, 132) == 0
    with pytest.raises(ValueError):
        attn.emulated_partitions("flashinfer", 1, 4, 100, 132)


def _args(**over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, lens=FAKE, o=FAKE, lse=None, N=2, Hq=8, Hkv=2, d=128, page=16,
             maxb=4, nblocks=8, numerics=3, parts=2, scale=0.1, ws=FAKE, wsb=1 << 20, stream=None)
    a.update(over)
    return tuple(a.values())


@pytest.mark.parametrize("over,want", [
    (dict(q=None), 1), (dict(bt=FAKE + 2), 1), (dict(N=0), 1), (dict(Hkv=3), 1), (dict(scale=0.0), 1),
    (dict(page=32), 2), (dict(d=64), 2),
    (dict(numerics=0), 1), (dict(numerics=5), 1), (dict(parts=0), 1), (dict(parts=70000), 1),
    (dict(ws=None), 3), (dict(wsb=10), 3), (dict(ws=FAKE + 4), 3),
])
def test_decode_emulated_argument_checks(attn, over, want):
    assert attn.lib().attn_decode_paged_emulated(*_args(**over)) == want


def test_merge_argument_checks(attn):
    lib = attn.lib()
    ok = dict(n=1, po=FAKE, pm=FAKE, pl=FAKE, rows=4, splits=3, d=128, o32=FAKE, o=FAKE, lse=None, stream=None)

    def call(**over):
        a = dict(ok)
        a.update(over)
        return lib.attn_merge_emulated(*a.values())

    assert call(n=0) == 1
    assert call(po=None) == 1
    assert call(o32=None, o=None) == 1
    assert call(pm=FAKE + 2) == 1
    assert call(o=FAKE + 1) == 1
    assert call(rows=0) == 1
    assert call(splits=0) == 1
    assert call(d=0) == 1
    assert call(d=1025) == 1
