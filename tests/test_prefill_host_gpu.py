"""attn_prefill_host: a prefill whose inputs and outputs are in host memory, with the transfers
inside the call, pipelined over query chunks.  Parity against the float64 oracle through the C ABI,
and equality with the device-resident attn_prefill on the same sequence."""
import math

import numpy as np
import pytest
import torch

import oracle.attention as oa
from parity import check_lse, check_o, to_np
from workloads import make_prefill_inputs

pytestmark = pytest.mark.gpu


def host_inputs(S, Hq, Hkv, d, seed, pin=True):
    x = make_prefill_inputs(1, Hq, Hkv, S, d, seed=seed)
    q, k, v = (t[0].contiguous() for t in (x.q, x.k, x.v))
    if pin:
        q, k, v = (t.pin_memory() for t in (q, k, v))
    return x, q, k, v


def run_host(attn, q, k, v, scale, causal, chunks, gpu, pin=True):
    S, Hq, d = q.shape
    o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, pin_memory=pin)
    lse = torch.full((Hq, S), float("nan"), dtype=torch.float32, pin_memory=pin)
    with torch.cuda.device(gpu):
        attn.prefill_host(q, k, v, scale=scale, causal=causal, chunks=chunks, out=o, lse=lse, device=gpu)
        torch.cuda.synchronize()
    return o, lse


@pytest.mark.parametrize("chunks", [1, 3, 4, 7])
def test_host_prefill_matches_oracle_and_device_prefill(attn, gpu, chunks):
    """1000 rows (not a multiple of the chunk count, the 16-token page or the 128-row tile), 4 query
    heads per KV head (CTA pairs): every output against the oracle, and bit for bit against
    attn_prefill on the device copies of the same inputs."""
    S, Hq, Hkv, d = 1000, 8, 2, 128
    scale = 1.0 / math.sqrt(d)
    x, q, k, v = host_inputs(S, Hq, Hkv, d, seed=120 + chunks)
    o, lse = run_host(attn, q, k, v, scale, True, chunks, gpu)
    wo, wl = oa.prefill(x.q, x.k, x.v, scale, causal=True)
    check_o(to_np(o)[None], wo, f"host prefill, {chunks} chunks")
    check_lse(to_np(lse)[None], wl, f"host prefill lse, {chunks} chunks")
    od, ld = attn.prefill(*(t.to(gpu) for t in (x.q, x.k, x.v)), scale=scale, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o, od[0].cpu()) and torch.equal(lse, ld[0].cpu())


@pytest.mark.parametrize("shape", [(6, 2, 64), (6, 2, 128), (4, 1, 256)], ids=["d64", "d128-odd-groups", "d256"])
@pytest.mark.parametrize("causal", [True, False])
def test_host_prefill_head_dims_and_masking(attn, gpu, shape, causal):
    """The single-CTA kernel's shapes (d = 64 and 256, 3 query heads per KV head), causal and not:
    without the causal mask every chunk sees all keys (k and v copied before the first chunk)."""
    Hq, Hkv, d = shape
    S = 333
    scale = 1.0 / math.sqrt(d)
    x, q, k, v = host_inputs(S, Hq, Hkv, d, seed=130 + d + causal)
    o, lse = run_host(attn, q, k, v, scale, causal, 3, gpu)
    wo, wl = oa.prefill(x.q, x.k, x.v, scale, causal=causal)
    check_o(to_np(o)[None], wo, f"host prefill d={d} causal={causal}")
    check_lse(to_np(lse)[None], wl, f"host prefill lse d={d} causal={causal}")


def test_host_prefill_pageable_and_repeated(attn, gpu):
    """Pageable host buffers give the same bits as page-locked ones; calls back to back on one
    stream, over one workspace, each see their own inputs."""
    S, Hq, Hkv, d = 700, 8, 2, 128
    scale = 0.1
    x, q, k, v = host_inputs(S, Hq, Hkv, d, seed=140)
    o_pin, l_pin = run_host(attn, q, k, v, scale, True, 4, gpu)
    o_pg, l_pg = run_host(attn, *(t.clone() for t in (q, k, v)), scale, True, 4, gpu, pin=False)
    assert not o_pg.is_pinned()
    assert torch.equal(o_pin, o_pg) and torch.equal(l_pin, l_pg)
    # three calls enqueued before one synchronisation, the inputs changing between them
    ws = torch.empty(attn.prefill_host_workspace_bytes(S, Hq, Hkv, d, 4), dtype=torch.uint8, device=gpu)
    outs = []
    ins = [host_inputs(S, Hq, Hkv, d, seed=141 + i) for i in range(3)]
    with torch.cuda.device(gpu):
        for xi, qi, ki, vi in ins:
            oi = torch.empty(qi.shape, dtype=torch.bfloat16, pin_memory=True)
            attn.prefill_host(qi, ki, vi, scale=scale, chunks=4, out=oi, return_lse=False, workspace=ws)
            outs.append(oi)
        torch.cuda.synchronize()
    for (xi, *_), oi in zip(ins, outs):
        wo, _ = oa.prefill(xi.q, xi.k, xi.v, scale, causal=True, heads=[0, 7])
        check_o(to_np(oi)[None][:, :, [0, 7]], wo[:, :, [0, 7]], "back-to-back host prefill")


def test_host_prefill_llama8b_cell(attn, gpu):
    """The Llama-8B cell (S = 2048, 32 query heads, 8 KV heads) in 4 chunks, as bench.py times it:
    bit for bit the device prefill, and sampled heads against the oracle."""
    S, Hq, Hkv, d = 2048, 32, 8, 128
    scale = 1.0 / math.sqrt(d)
    x, q, k, v = host_inputs(S, Hq, Hkv, d, seed=150)
    o, lse = run_host(attn, q, k, v, scale, True, 4, gpu)
    od, ld = attn.prefill(*(t.to(gpu) for t in (x.q, x.k, x.v)), scale=scale, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o, od[0].cpu()) and torch.equal(lse, ld[0].cpu())
    heads = [0, 13, 31]
    wo, wl = oa.prefill(x.q, x.k, x.v, scale, causal=True, heads=heads)
    check_o(to_np(o)[None][:, :, heads], wo[:, :, heads], "host prefill llama8b")
    check_lse(to_np(lse)[None][:, heads], wl[:, heads], "host prefill llama8b lse")
