"""The allocation-free paged decode matches the regular one and the oracle.

attn_decode_paged_noalloc serves callers that cannot hand the library a
workspace (a plugin whose host framework owns all device memory, a serving
loop that forbids device allocations after start-up): its split partials live
in a fixed array inside the library.  Here it is called several times in a
row, through the C ABI and through the Python wrapper, on different inputs and
split settings (balanced mode included), and each result is compared both
with attn_decode_paged given a caller-allocated workspace and with the
float64 oracle.  A later call over shorter sequences reuses the slot layout
of an earlier, longer one, so slots that the earlier call filled are left
over in the array; they must not leak into the result.  This file is
collected last so that a failure here cannot hide any other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle.attention as oa
from parity import check_lse, check_o, to_np
from workloads import make_decode_inputs

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20   # ATTN_DECODE_NOALLOC_SCRATCH_BYTES in include/attn.h


def _noalloc_c_abi(attn, x, scale, num_splits, split_tokens, dev):
    """Call attn_decode_paged_noalloc directly through ctypes."""
    q, kc, vc, bt, sl = (t.to(dev) for t in (x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens))
    N, Hq, d = q.shape
    num_blocks, page, Hkv, _ = kc.shape
    o = torch.full_like(q, float("nan"))
    lse = torch.full((N, Hq), float("nan"), dtype=torch.float32, device=dev)
    fn = attn.lib().attn_decode_paged_noalloc
    st = fn(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), sl.data_ptr(), o.data_ptr(), lse.data_ptr(),
            N, Hq, Hkv, d, page, bt.shape[1], num_blocks, num_splits, split_tokens, ctypes.c_float(scale),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st, o, lse


def _noalloc_python(attn, x, scale, num_splits, split_tokens, dev):
    args = [t.to(dev) for t in (x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens)]
    o, lse = attn.decode_paged_noalloc(*args, scale=scale, num_splits=num_splits, split_tokens=split_tokens)
    torch.cuda.synchronize()
    return 0, o, lse


def _regular(attn, x, scale, num_splits, split_tokens, dev):
    args = [t.to(dev) for t in (x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens)]
    o, lse = attn.decode_paged(*args, scale=scale, num_splits=num_splits, split_tokens=split_tokens)
    torch.cuda.synchronize()
    return o, lse


def _check_against_both(attn, x, scale, ns, span, o, lse, dev, what):
    live = x.seq_lens.numpy() > 0
    ro, rl = _regular(attn, x, scale, ns, span, dev)
    check_o(to_np(o), to_np(ro), f"{what} vs attn_decode_paged")
    check_lse(to_np(lse)[live], to_np(rl)[live], f"{what} vs attn_decode_paged")
    # an empty sequence: o = 0 and lse = -inf, as the regular call gives
    assert (to_np(o)[~live] == 0).all() and np.isneginf(to_np(lse)[~live]).all(), what
    wo, wl = oa.decode_paged(x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens, scale)
    check_o(to_np(o)[live], wo[live], f"{what} vs oracle")
    check_lse(to_np(lse)[live], wl[live], f"{what} vs oracle")


def test_noalloc_matches_regular_and_oracle_in_a_row(attn, gpu):
    long_lens = [1, 40, 300, 1000, 2047]
    x_long = make_decode_inputs(long_lens, Hq=32, Hkv=8, d=128, seed=71, nan_tail=True)
    # the same slot layout (block-table width, split count) as x_long, over shorter sequences: the later
    # groups of every sequence are empty in this call but were filled by the first one
    x_short = make_decode_inputs([1, 17, 33, 200, 64], Hq=32, Hkv=8, d=128, seed=74, nan_tail=True)
    wide = torch.zeros_like(x_long.block_table)
    wide[:, :x_short.block_table.shape[1]] = x_short.block_table
    x_short.block_table = wide
    calls = [
        (_noalloc_c_abi, x_long, 0.09, 16, 0),
        (_noalloc_c_abi, make_decode_inputs([700, 5000, 12], Hq=16, Hkv=2, d=256, seed=72, nan_tail=True),
         2.0 ** -4, 1, 512),
        (_noalloc_python, x_short, 0.09, 16, 0),
        # balanced mode (num_splits = split_tokens = 0), twice on different lengths
        (_noalloc_c_abi, make_decode_inputs([3000, 9, 450], Hq=16, Hkv=2, d=256, seed=75, nan_tail=True),
         2.0 ** -4, 0, 0),
        (_noalloc_python, make_decode_inputs([5, 800, 0, 2500], Hq=8, Hkv=2, d=128, seed=76, nan_tail=True),
         0.1, 0, 0),
    ]
    for i, (call, x, scale, ns, span) in enumerate(calls):
        st, o, lse = call(attn, x, scale, ns, span, gpu)
        assert st == 0, f"call {i}: status {st}"
        _check_against_both(attn, x, scale, ns, span, o, lse, gpu, f"no-alloc call {i}")


def test_noalloc_rejects_too_large(attn, gpu):
    """Partials beyond the fixed array are refused before anything is enqueued."""
    x = make_decode_inputs([64] * 4, Hq=32, Hkv=8, d=256, seed=73)
    N, Hq, d = x.q.shape
    # enough splits that N * Hq * splits * (d + 2) * 4 bytes exceed the array
    splits = SCRATCH_BYTES // (N * Hq * (d + 2) * 4) + 1
    bt = torch.zeros((N, splits), dtype=torch.int32)
    bt[:, :4] = x.block_table[:, :4]
    x.block_table = bt
    st, o, _ = _noalloc_c_abi(attn, x, 0.06, splits, 0, gpu)
    assert st == 3                                   # ATTN_ERR_WORKSPACE
    assert torch.isnan(o).all()                      # nothing ran
    # an argument error is reported as such, even when the partials would not fit either
    st, o, _ = _noalloc_c_abi(attn, x, -1.0, splits, 0, gpu)
    assert st == 1                                   # ATTN_ERR_INVALID_ARG (non-positive scale)
    assert torch.isnan(o).all()
