"""Packed-sequence (varlen) prefill parity through the C ABI against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle.attention as oa
from parity import check_lse, check_o, to_np
from workloads import make_prefill_inputs, make_varlen_inputs

pytestmark = pytest.mark.gpu

SENTINEL = 7.0  # exactly representable in bf16; rows that belong to no sequence keep it


def run_varlen(attn, x, scale, causal, dev):
    q, k, v, cu = (t.to(dev) for t in (x.q, x.k, x.v, x.cu_seqlens))
    out = torch.full_like(q, SENTINEL)
    lse = torch.full((q.shape[1], q.shape[0]), SENTINEL, dtype=torch.float32, device=dev)
    attn.prefill_varlen(q, k, v, cu, x.max_seqlen, scale=scale, causal=causal, out=out, lse=lse)
    torch.cuda.synchronize()
    return out, lse


def compare(attn, x, scale, causal, dev, what, seqs=None, heads=None):
    o, lse = run_varlen(attn, x, scale, causal, dev)
    wo, wl = oa.prefill_varlen(x.q, x.k, x.v, x.cu_seqlens, scale, causal=causal, seqs=seqs, heads=heads)
    cu = x.cu_seqlens.tolist()
    seqs = range(len(cu) - 1) if seqs is None else seqs
    heads = list(range(x.q.shape[1])) if heads is None else list(heads)
    rows = np.concatenate([np.arange(cu[n], cu[n + 1]) for n in seqs] + [np.zeros(0, np.int64)]).astype(np.int64)
    if rows.size:
        check_o(to_np(o)[rows][:, heads], wo[rows][:, heads], what)
        check_lse(to_np(lse)[heads][:, rows], wl[heads][:, rows], what)
    return o, lse


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_ragged_pack(attn, gpu, causal, d):
    """Lengths around tile edges, an empty sequence, GQA 4:2, two trailing tokens in no sequence."""
    lens = [1, 127, 0, 128, 129, 300, 7, 513]
    x = make_varlen_inputs(lens, Hq=4, Hkv=2, d=d, seed=70 + d + causal, extra=2)
    o, lse = compare(attn, x, 1.0 / math.sqrt(d), causal, gpu, f"varlen d={d} causal={causal}")
    assert torch.all(o[-2:].float() == SENTINEL) and torch.all(lse[:, -2:] == SENTINEL)


def test_equal_lengths_match_fixed_batch(attn, gpu):
    """N packed sequences of S tokens give the fixed-length batch result bit for bit."""
    B, S, Hq, Hkv, d = 3, 300, 4, 2, 128
    x = make_prefill_inputs(B, Hq, Hkv, S, d, seed=77)
    q, k, v = (t.to(gpu) for t in (x.q, x.k, x.v))
    of, lf = attn.prefill(q, k, v, scale=0.088, causal=True)
    cu = torch.arange(0, (B + 1) * S, S, dtype=torch.int32, device=gpu)
    ov, lv = attn.prefill_varlen(q.reshape(B * S, Hq, d), k.reshape(B * S, Hkv, d), v.reshape(B * S, Hkv, d), cu, S,
                                 scale=0.088, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(ov.reshape(B, S, Hq, d), of)
    assert torch.equal(lv.reshape(Hq, B, S).permute(1, 0, 2), lf)


def test_many_short_sequences(attn, gpu):
    """More sequences than SMs, most shorter than one tile (the tile list skips empty levels)."""
    rng = np.random.default_rng(78)
    lens = [int(x) for x in rng.integers(0, 200, size=400)]
    x = make_varlen_inputs(lens, Hq=2, Hkv=1, d=64, seed=78)
    compare(attn, x, 0.125, True, gpu, "400 short sequences", seqs=range(0, 400, 7))


def test_mixed_long_sequences_sampled(attn, gpu):
    """Llama-8B heads, lengths 37 .. 4096 packed; sampled sequences and heads."""
    lens = [2048, 1000, 37, 4096, 513]
    x = make_varlen_inputs(lens, Hq=32, Hkv=8, d=128, seed=79)
    compare(attn, x, 1.0 / math.sqrt(128), True, gpu, "mixed lengths", seqs=[1, 2, 4], heads=[0, 13, 31])


@pytest.mark.parametrize("heads", [(2, 1, 64), (4, 2, 128)], ids=["single-CTA", "CTA-pair"])
def test_bad_offsets_are_reported(attn, gpu, heads):
    """Offsets past the tokens or running backwards are recorded as device status 5 and skipped."""
    Hq, Hkv, d = heads
    lens = [40, 60, 30]
    x = make_varlen_inputs(lens, Hq=Hq, Hkv=Hkv, d=d, seed=80)
    cu = x.cu_seqlens.clone()
    cu[2] = 200                  # sequence 1 ends past the 130 tokens, sequence 2 runs backwards
    x2 = type(x)(x.q, x.k, x.v, cu, 0)
    o, _ = run_varlen(attn, x2, 0.125, True, gpu)
    assert attn.device_status(clear=True) == 5
    assert torch.all(o[40:].float() == SENTINEL)  # the skipped sequences' rows are not written
    compare(attn, x2, 0.125, True, gpu, "valid sequence", seqs=[0])
    attn.device_status(clear=True)
