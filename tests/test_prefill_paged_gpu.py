"""Chunked prefill against the paged cache: parity through the C ABI against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle.attention as oa
from parity import check_lse, check_o, to_np
from workloads import make_chunked_inputs, make_prefill_inputs, prefill_inputs_for

pytestmark = pytest.mark.gpu

SENTINEL = 7.0


def run(attn, x, scale, causal, dev):
    args = [t.to(dev) for t in (x.q, x.k_cache, x.v_cache, x.block_table, x.cu_seqlens_q, x.seq_lens)]
    out = torch.full_like(args[0], SENTINEL)
    lse = torch.full((x.q.shape[1], x.q.shape[0]), SENTINEL, dtype=torch.float32, device=dev)
    attn.prefill_paged(*args, x.max_seqlen_q, scale=scale, causal=causal, out=out, lse=lse)
    torch.cuda.synchronize()
    return out, lse


def compare(attn, x, scale, causal, dev, what, seqs=None, heads=None):
    o, lse = run(attn, x, scale, causal, dev)
    wo, wl = oa.prefill_paged(x.q, x.k_cache, x.v_cache, x.block_table, x.cu_seqlens_q, x.seq_lens, scale,
                              causal=causal, seqs=seqs, heads=heads)
    cu = x.cu_seqlens_q.tolist()
    seqs = range(len(cu) - 1) if seqs is None else seqs
    heads = list(range(x.q.shape[1])) if heads is None else list(heads)
    rows = np.concatenate([np.arange(cu[n], cu[n + 1]) for n in seqs] + [np.zeros(0, np.int64)]).astype(np.int64)
    if rows.size:
        check_o(to_np(o)[rows][:, heads], wo[rows][:, heads], what)
        check_lse(to_np(lse)[heads][:, rows], wl[heads][:, rows], what)
    return o, lse


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_chunks_over_cached_context(attn, gpu, causal, d):
    """Chunks of 1..300 new tokens over 1..1000 cached ones; NaN in page tails and in unused pages."""
    ctx = [100, 300, 1000, 17, 129, 640, 33]
    ql = [100, 1, 37, 0, 128, 300, 32]
    x = make_chunked_inputs(ctx, ql, Hq=4, Hkv=2, d=d, seed=90 + d + causal, nan_tail=True, extra_blocks=4)
    compare(attn, x, 1.0 / math.sqrt(d), causal, gpu, f"chunked d={d} causal={causal}")


def test_whole_prompt_chunk_equals_prefill(attn, gpu):
    """A chunk that is the whole sequence, with the cache pages in order, gives the contiguous prefill bit for bit."""
    B, S, Hq, Hkv, d = 1, 300, 4, 2, 128
    x = make_prefill_inputs(B, Hq, Hkv, S, d, seed=91)
    pages = (S + 15) // 16
    kc = torch.zeros((pages, 16, Hkv, d), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    kc.view(-1, Hkv, d)[:S] = x.k[0]
    vc.view(-1, Hkv, d)[:S] = x.v[0]
    bt = torch.arange(pages, dtype=torch.int32)[None]
    q, kc, vc, bt = (t.to(gpu) for t in (x.q[0], kc, vc, bt))
    cu = torch.tensor([0, S], dtype=torch.int32, device=gpu)
    sl = torch.tensor([S], dtype=torch.int32, device=gpu)
    op, lp = attn.prefill_paged(q, kc, vc, bt, cu, sl, S, scale=0.09, causal=True)
    of, lf = attn.prefill(*(t.to(gpu) for t in (x.q, x.k, x.v)), scale=0.09, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(op, of[0]) and torch.equal(lp, lf[0])


def test_long_context_chunks_sampled(attn, gpu):
    """Llama-8B heads: 2048-token chunks over 2K..16K cached tokens; sampled sequences and heads."""
    ctx = [4096, 16384, 2048, 9000]
    ql = [2048, 2048, 2048, 1000]
    x = make_chunked_inputs(ctx, ql, Hq=32, Hkv=8, d=128, seed=92)
    compare(attn, x, 1.0 / math.sqrt(128), True, gpu, "long chunks", seqs=[1, 3], heads=[0, 9, 31])


@pytest.mark.parametrize("Hq", [8, 6], ids=["CTA-pair", "single-CTA"])
def test_chunks_over_more_context_than_l2(attn, gpu, Hq):
    """Nineteen sequences whose cached keys and values (4 MB a sequence at the block table's 4096
    tokens, about 80 MB in all) exceed half of L2: the walk takes them in blocks of a few sequences,
    the last block partial; every sequence is checked, in both kernels (4 and 3 query heads per KV
    head)."""
    ctx = [4096, 3000, 4096, 2500, 4096, 3900, 4096, 2048, 4096, 3333, 4096, 1, 4000, 4096, 700, 4096, 2222, 4096, 3500]
    ql = [512, 300, 512, 257, 512, 400, 128, 512, 1, 333, 512, 1, 129, 64, 700, 200, 17, 511, 256]
    x = make_chunked_inputs(ctx, ql, Hq=Hq, Hkv=2, d=128, seed=94)
    compare(attn, x, 1.0 / math.sqrt(128), True, gpu, "blocked walk", heads=[0, 5, Hq - 1])


@pytest.mark.parametrize("heads", [(2, 1, 64), (4, 2, 128)], ids=["single-CTA", "CTA-pair"])
def test_bad_page_and_bad_lengths_are_reported(attn, gpu, heads):
    Hq, Hkv, d = heads
    x = make_chunked_inputs([40, 50], [10, 50], Hq=Hq, Hkv=Hkv, d=d, seed=93)
    bt = x.block_table.clone()
    bt[0, 1] = x.k_cache.shape[0] + 5
    x2 = type(x)(x.q, x.k_cache, x.v_cache, bt, x.seq_lens, x.cu_seqlens_q)
    run(attn, x2, 0.125, True, gpu)
    assert attn.device_status(clear=True) == 2
    sl = x.seq_lens.clone()
    sl[1] = 30                                   # fewer cached tokens than new ones
    x3 = type(x)(x.q, x.k_cache, x.v_cache, x.block_table, sl, x.cu_seqlens_q)
    o, _ = run(attn, x3, 0.125, True, gpu)
    assert attn.device_status(clear=True) == 5
    assert torch.all(o[10:].float() == SENTINEL)
    compare(attn, x3, 0.125, True, gpu, "valid sequence", seqs=[0])
    attn.device_status(clear=True)
