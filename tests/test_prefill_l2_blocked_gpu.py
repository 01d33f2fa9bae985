"""Equal-length batches whose keys and values exceed three quarters of L2 (d = 128) or one and a half
times L2 (d = 64 and 256): the blocked walk.

Such batches are walked in blocks of whole KV heads, (sequence, KV head) lanes whose keys and values
take at most an eighth of L2, band by band of query-tile levels.  The order of the walk cannot change a
tile's arithmetic, so the output must equal, bit for bit, the same batch computed as slices of a few
KV heads each (small enough for the plain walk); sampled rows of a few heads are also checked
against the float64 oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle.attention as oa
from parity import check_lse, check_o, to_np
from workloads import make_prefill_inputs, make_varlen_inputs

pytestmark = pytest.mark.gpu


def sliced(attn, q, k, v, scale, kv_per_slice):
    """The prefill of every slice of kv_per_slice KV heads (and their query heads) on its own."""
    B, S, Hq, d = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    for g0 in range(0, Hkv, kv_per_slice):
        g1 = min(Hkv, g0 + kv_per_slice)
        qs = q[:, :, g0 * G:g1 * G].contiguous()
        os_, ls = attn.prefill(qs, k[:, :, g0:g1].contiguous(), v[:, :, g0:g1].contiguous(), scale=scale,
                               causal=True)
        o[:, :, g0 * G:g1 * G] = os_
        lse[:, g0 * G:g1 * G] = ls
    return o, lse


@pytest.mark.parametrize("shape", [(4, 32, 32, 4096, 128, 4), (6, 32, 8, 8192, 128, 1), (3, 24, 24, 4096, 128, 3),
                                   (4, 32, 32, 8192, 64, 4), (2, 16, 16, 8192, 256, 2)],
                         ids=["mha-single-CTA", "gqa-CTA-pairs", "mha-partial-last-block", "mha-d64", "mha-d256"])
def test_blocked_walk_equals_slices_and_oracle(attn, gpu, shape):
    B, Hq, Hkv, S, d, kv_per_slice = shape
    assert S * d * 4 * B * Hkv > 130 * 2 ** 20         # more than L2: the blocked walk at d = 128
    assert S * d * 4 * B * kv_per_slice < 40 * 2 ** 20  # a slice: the plain walk
    x = make_prefill_inputs(B, Hq, Hkv, S, d, seed=8800 + d + Hkv)
    scale = 1.0 / math.sqrt(d)
    q, k, v = (t.to(gpu) for t in (x.q, x.k, x.v))
    o, lse = attn.prefill(q, k, v, scale=scale, causal=True)
    os_, ls = sliced(attn, q, k, v, scale, kv_per_slice)
    torch.cuda.synchronize()
    assert torch.equal(o, os_) and torch.equal(lse, ls)
    heads = [0, Hq // 2 + 1, Hq - 1]
    rows = np.array([0, 1, 127, 128, S // 2 - 1, S // 2, S - 129, S - 1])
    r_t, h_t = torch.tensor(rows, device=gpu), torch.tensor(heads, device=gpu)
    for b in sorted({0, B - 1}):
        wo, wl = oa.prefill(x.q, x.k, x.v, scale, causal=True, heads=heads, rows=rows, batches=[b])
        check_o(to_np(o[b][r_t][:, h_t]), wo[b][rows][:, heads], f"blocked walk b={b}")
        check_lse(to_np(lse[b][h_t][:, r_t]), wl[b][heads][:, rows], f"blocked walk b={b}")


def test_packed_equal_lengths_blocked_equals_equal_length_call(attn, gpu):
    """Packed prompts larger than L2 (8 x 4096 tokens, 32 query and 32 KV heads: single-CTA kernel):
    the packed blocked walk gives the equal-length call's output bit for bit."""
    B, H, S, d = 8, 32, 4096, 128
    x = make_prefill_inputs(B, H, H, S, d, seed=8900)
    scale = 1.0 / math.sqrt(d)
    q, k, v = (t.to(gpu) for t in (x.q, x.k, x.v))
    o, lse = attn.prefill(q, k, v, scale=scale, causal=True)
    cu = torch.arange(0, (B + 1) * S, S, dtype=torch.int32, device=gpu)
    op, lp = attn.prefill_varlen(q.view(B * S, H, d), k.view(B * S, H, d), v.view(B * S, H, d), cu, S, scale=scale,
                                 causal=True)
    torch.cuda.synchronize()
    assert torch.equal(op.view(B, S, H, d), o)
    assert torch.equal(lp.view(H, B, S).transpose(0, 1), lse)


def test_packed_ragged_blocked_equals_small_groups_and_oracle(attn, gpu):
    """A ragged pack larger than L2 (12 prompts of 1-8K tokens, 32 query / 8 KV heads: CTA pairs)
    against the same prompts run as packs of three (each small enough for the plain walk), bit for
    bit, and sampled rows against the oracle."""
    rng = np.random.default_rng(8901)
    lens = [int(v) for v in rng.integers(1024, 8193, size=12)]
    lens[3] = 8192
    Hq, Hkv, d = 32, 8, 128
    x = make_varlen_inputs(lens, Hq=Hq, Hkv=Hkv, d=d, seed=8902)
    assert sum(lens) * Hkv * d * 4 > 130 * 2 ** 20
    scale = 1.0 / math.sqrt(d)
    q, k, v, cu = (t.to(gpu) for t in (x.q, x.k, x.v, x.cu_seqlens))
    o, lse = attn.prefill_varlen(q, k, v, cu, max(lens), scale=scale, causal=True)
    offs = x.cu_seqlens.tolist()
    o2, l2 = torch.empty_like(o), torch.empty_like(lse)
    for g0 in range(0, len(lens), 3):
        g1 = min(len(lens), g0 + 3)
        a, b = offs[g0], offs[g1]
        cug = torch.tensor([t - a for t in offs[g0:g1 + 1]], dtype=torch.int32, device=gpu)
        og, lg = attn.prefill_varlen(q[a:b].contiguous(), k[a:b].contiguous(), v[a:b].contiguous(), cug,
                                     max(lens[g0:g1]), scale=scale, causal=True)
        o2[a:b], l2[:, a:b] = og, lg
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, l2)
    heads = [0, 17, 31]
    for n in (0, 3, len(lens) - 1):
        rows = np.array([0, 1, 128, lens[n] // 2, lens[n] - 1]) + offs[n]
        wo, wl = oa.prefill_varlen(x.q, x.k, x.v, x.cu_seqlens, scale, causal=True, heads=heads, seqs=[n])
        r_t, h_t = torch.tensor(rows, device=gpu), torch.tensor(heads, device=gpu)
        check_o(to_np(o[r_t][:, h_t]), wo[rows][:, heads], f"packed blocked seq {n}")
        check_lse(to_np(lse[h_t][:, r_t]), wl[heads][:, rows], f"packed blocked seq {n}")
