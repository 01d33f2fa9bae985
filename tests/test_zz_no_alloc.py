"""The allocation-free paged decode matches the regular one.

attn_decode_paged_noalloc serves callers that cannot hand the library a
workspace (a plugin whose host framework owns all device memory, a serving
loop that forbids device allocations after start-up): its split partials live
in a fixed array inside the library.  Here it is called through the C ABI
twice in a row, on different inputs and split settings, and each result is
compared with attn_decode_paged given a caller-allocated workspace.  This file
is collected last so that a failure here cannot hide any other test.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

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


def _regular(attn, x, scale, num_splits, split_tokens, dev):
    args = [t.to(dev) for t in (x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens)]
    o, lse = attn.decode_paged(*args, scale=scale, num_splits=num_splits, split_tokens=split_tokens)
    torch.cuda.synchronize()
    return o, lse


def test_noalloc_matches_regular_twice(attn, gpu):
    calls = [
        (make_decode_inputs([1, 40, 300, 1000, 2047], Hq=32, Hkv=8, d=128, seed=71, nan_tail=True), 0.09, 4, 0),
        (make_decode_inputs([700, 5000, 12], Hq=16, Hkv=2, d=256, seed=72, nan_tail=True), 2.0 ** -4, 1, 512),
    ]
    for i, (x, scale, ns, span) in enumerate(calls):
        st, o, lse = _noalloc_c_abi(attn, x, scale, ns, span, gpu)
        assert st == 0, f"call {i}: status {st}"
        ro, rl = _regular(attn, x, scale, ns, span, gpu)
        check_o(to_np(o), to_np(ro), f"no-alloc call {i}")
        check_lse(to_np(lse), to_np(rl), f"no-alloc call {i}")


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
