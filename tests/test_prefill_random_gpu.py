"""Seeded random shapes through every prefill entry point, against the float64 oracle.

Each seed draws a batch shape (lengths around tile and page edges and long ones, 1 to 8 query heads per
KV head, head dim 64 / 128 / 256, causal or not) and runs it through attn_prefill, attn_prefill_varlen,
attn_prefill_paged or attn_prefill_host; every output row of every head is compared.  The shapes reach
both kernels (CTA pairs at d = 128 with even head groups, single CTAs otherwise) and their ragged,
packed, paged and chunked forms, and batches large enough for the blocked walk.
"""

import numpy as np
import pytest
import torch

import oracle.attention as oa
from parity import check_lse, check_o, to_np
from workloads import make_chunked_inputs, make_prefill_inputs, make_varlen_inputs

pytestmark = pytest.mark.gpu

EDGE_LENS = [1, 2, 15, 16, 17, 127, 128, 129, 255, 256, 257, 383, 640, 1000, 1500]
HEADS = [(1, 1), (2, 1), (3, 1), (4, 2), (6, 6), (8, 1), (8, 2), (12, 4), (16, 2)]


def draw(seed):
    rng = np.random.default_rng(7000 + seed)
    Hq, Hkv = HEADS[int(rng.integers(0, len(HEADS)))]
    d = [64, 128, 256][int(rng.integers(0, 3))]
    causal = bool(rng.integers(0, 4))  # mostly causal
    return rng, Hq, Hkv, d, causal


def rows_of(cu, seqs):
    return np.concatenate([np.arange(cu[n], cu[n + 1]) for n in seqs] + [np.zeros(0, np.int64)]).astype(np.int64)


@pytest.mark.parametrize("seed", range(8))
def test_random_equal_length_batches(attn, gpu, seed):
    rng, Hq, Hkv, d, causal = draw(seed)
    B = int(rng.integers(1, 4))
    S = int(rng.choice(EDGE_LENS))
    x = make_prefill_inputs(B, Hq, Hkv, S, d, seed=7100 + seed)
    scale = float(d) ** -0.5
    o, lse = attn.prefill(*(t.to(gpu) for t in (x.q, x.k, x.v)), scale=scale, causal=causal)
    torch.cuda.synchronize()
    wo, wl = oa.prefill(x.q, x.k, x.v, scale, causal=causal)
    what = f"seed {seed}: B={B} S={S} Hq={Hq} Hkv={Hkv} d={d} causal={causal}"
    check_o(to_np(o), wo, what)
    check_lse(to_np(lse), wl, what)


@pytest.mark.parametrize("seed", range(8))
def test_random_packed_sequences(attn, gpu, seed):
    rng, Hq, Hkv, d, causal = draw(seed + 100)
    N = int(rng.integers(1, 9))
    lens = [int(v) for v in rng.choice(EDGE_LENS + [0], size=N)]
    if sum(lens) == 0:
        lens[0] = 33
    x = make_varlen_inputs(lens, Hq=Hq, Hkv=Hkv, d=d, seed=7200 + seed, extra=int(rng.integers(0, 3)))
    scale = float(d) ** -0.5
    q, k, v, cu = (t.to(gpu) for t in (x.q, x.k, x.v, x.cu_seqlens))
    o = torch.zeros_like(q)  # rows of no sequence are not written
    lse = torch.zeros((Hq, q.shape[0]), dtype=torch.float32, device=gpu)
    attn.prefill_varlen(q, k, v, cu, x.max_seqlen, scale=scale, causal=causal, out=o, lse=lse)
    torch.cuda.synchronize()
    wo, wl = oa.prefill_varlen(x.q, x.k, x.v, x.cu_seqlens, scale, causal=causal)
    rows = rows_of(x.cu_seqlens.tolist(), range(N))
    what = f"seed {seed}: lens={lens} Hq={Hq} Hkv={Hkv} d={d} causal={causal}"
    check_o(to_np(o)[rows], wo[rows], what)
    check_lse(to_np(lse)[:, rows], wl[:, rows], what)


@pytest.mark.parametrize("seed", range(8))
def test_random_chunks_over_paged_caches(attn, gpu, seed):
    rng, Hq, Hkv, d, causal = draw(seed + 200)
    N = int(rng.integers(1, 7))
    ctx = [int(v) for v in rng.choice(EDGE_LENS + [3000], size=N)]
    ql = [int(rng.integers(1, c + 1)) if rng.integers(0, 3) else c for c in ctx]  # a third whole prompts
    x = make_chunked_inputs(ctx, ql, Hq=Hq, Hkv=Hkv, d=d, seed=7300 + seed, nan_tail=True,
                            extra_blocks=int(rng.integers(0, 4)))
    scale = float(d) ** -0.5
    args = [t.to(gpu) for t in (x.q, x.k_cache, x.v_cache, x.block_table, x.cu_seqlens_q, x.seq_lens)]
    o, lse = attn.prefill_paged(*args, max(ql), scale=scale, causal=causal)
    torch.cuda.synchronize()
    wo, wl = oa.prefill_paged(x.q, x.k_cache, x.v_cache, x.block_table, x.cu_seqlens_q, x.seq_lens, scale,
                              causal=causal)
    rows = rows_of(x.cu_seqlens_q.tolist(), range(N))
    what = f"seed {seed}: ctx={ctx} q={ql} Hq={Hq} Hkv={Hkv} d={d} causal={causal}"
    check_o(to_np(o)[rows], wo[rows], what)
    check_lse(to_np(lse)[:, rows], wl[:, rows], what)


@pytest.mark.parametrize("seed", range(4))
def test_random_host_buffer_prefill(attn, gpu, seed):
    rng, Hq, Hkv, d, causal = draw(seed + 300)
    S = int(rng.choice(EDGE_LENS))
    chunks = int(rng.integers(1, 9))
    x = make_prefill_inputs(1, Hq, Hkv, S, d, seed=7400 + seed)
    scale = float(d) ** -0.5
    q, k, v = (t[0].contiguous().pin_memory() for t in (x.q, x.k, x.v))
    with torch.cuda.device(gpu):
        o, lse = attn.prefill_host(q, k, v, scale=scale, causal=causal, chunks=chunks, device=gpu)
        torch.cuda.synchronize()
    wo, wl = oa.prefill(x.q, x.k, x.v, scale, causal=causal)
    what = f"seed {seed}: S={S} chunks={chunks} Hq={Hq} Hkv={Hkv} d={d} causal={causal}"
    check_o(to_np(o)[None], wo, what)
    check_lse(to_np(lse)[None], wl, what)


@pytest.mark.parametrize("seed", range(6))
def test_random_batches_larger_than_l2(attn, gpu, seed):
    """Equal-length batches grown until their keys and values pass the blocked walk's threshold for the
    head dim (three quarters of L2 at d = 128, one and a half times at d = 64 and 256): bit for bit the
    same batch computed one KV head at a time, and sampled rows against the oracle."""
    rng, _, _, d, causal = draw(seed + 400)
    Hq, Hkv = [(8, 8), (32, 8), (32, 32), (12, 4), (24, 8), (16, 2)][int(rng.integers(0, 6))]
    S = int(rng.choice([2048, 4096, 8192]))
    l2 = torch.cuda.get_device_properties(gpu).L2_cache_size
    need = (0.8 if d == 128 else 1.6) * l2
    B = 1
    while S * d * 4 * B * Hkv < need:
        B += 1
    x = make_prefill_inputs(B, Hq, Hkv, S, d, seed=7500 + seed)
    scale = float(d) ** -0.5
    q, k, v = (t.to(gpu) for t in (x.q, x.k, x.v))
    o, lse = attn.prefill(q, k, v, scale=scale, causal=causal)
    G = Hq // Hkv
    for g in range(Hkv):
        og, lg = attn.prefill(q[:, :, g * G:(g + 1) * G].contiguous(), k[:, :, g:g + 1].contiguous(),
                              v[:, :, g:g + 1].contiguous(), scale=scale, causal=causal)
        assert torch.equal(o[:, :, g * G:(g + 1) * G], og) and torch.equal(lse[:, g * G:(g + 1) * G], lg), g
    torch.cuda.synchronize()
    rows = np.array([0, 1, S // 3, S // 2, S - 1])
    heads = sorted({0, Hq // 2, Hq - 1})
    b = int(rng.integers(0, B))
    wo, wl = oa.prefill(x.q, x.k, x.v, scale, causal=causal, heads=heads, rows=rows, batches=[b])
    r_t, h_t = torch.tensor(rows, device=gpu), torch.tensor(heads, device=gpu)
    what = f"seed {seed}: B={B} S={S} Hq={Hq} Hkv={Hkv} d={d} causal={causal}"
    check_o(to_np(o[b][r_t][:, h_t]), wo[b][rows][:, heads], what)
    check_lse(to_np(lse[b][h_t][:, r_t]), wl[b][heads][:, rows], what)
