"""Prefill parity: the tcgen05/TMA kernel (through the C ABI) against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle.attention as oa
from parity import check_lse, check_o, to_np
from workloads import LLAMA8B, QWEN256, SWEEP, TINY, make_prefill_inputs, prefill_inputs_for

pytestmark = pytest.mark.gpu


def run_prefill(attn, x, scale, causal, dev):
    q, k, v = (t.to(dev) for t in (x.q, x.k, x.v))
    o, lse = attn.prefill(q, k, v, scale=scale, causal=causal)
    torch.cuda.synchronize()
    return o, lse


def full_compare(attn, x, scale, causal, dev, what):
    o, lse = run_prefill(attn, x, scale, causal, dev)
    wo, wl = oa.prefill(x.q, x.k, x.v, scale, causal=causal)
    e = check_o(to_np(o), wo, what)
    check_lse(to_np(lse), wl, what)
    return e


def test_tiny_config(attn, gpu):
    """B=1, Hq=Hkv=1, S=128, d=64, scale=1/8: every output and LSE."""
    x = prefill_inputs_for(TINY)
    full_compare(attn, x, TINY.scale, True, gpu, "tiny")


@pytest.mark.parametrize("S", [1, 7, 128, 129, 255, 256, 257, 300, 511, 640])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_ragged_lengths_causal(attn, gpu, S, d):
    """Several Q/KV tiles with a ragged tail, GQA 4:2, two batch elements."""
    x = make_prefill_inputs(2, 4, 2, S, d, seed=1000 + S + d)
    full_compare(attn, x, 1.0 / math.sqrt(d), True, gpu, f"S={S} d={d}")


@pytest.mark.parametrize("S", [1, 100, 128, 300, 513])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_noncausal(attn, gpu, S, d):
    x = make_prefill_inputs(1, 2, 1, S, d, seed=2000 + S + d)
    full_compare(attn, x, 1.0 / math.sqrt(d), False, gpu, f"noncausal S={S} d={d}")


@pytest.mark.parametrize("S", [1, 129, 300, 640])
@pytest.mark.parametrize("Hq,Hkv", [(3, 1), (6, 2)])
def test_single_head_kernel_odd_groups(attn, gpu, S, Hq, Hkv):
    """Odd query heads per KV head at d = 128: the single-head kernel (pairs need an even group)."""
    x = make_prefill_inputs(2, Hq, Hkv, S, 128, seed=3000 + S + Hq)
    full_compare(attn, x, 1.0 / math.sqrt(128), True, gpu, f"odd groups Hq={Hq} Hkv={Hkv} S={S}")


@pytest.mark.parametrize("S", [1, 127, 128, 129, 1000])
@pytest.mark.parametrize("Hq,Hkv", [(2, 1), (8, 2), (16, 2)])
def test_pair_kernel_groups(attn, gpu, S, Hq, Hkv):
    """Even query heads per KV head at d = 128: CTA pairs, including one work unit and ragged tails."""
    x = make_prefill_inputs(1, Hq, Hkv, S, 128, seed=4000 + S + Hq)
    full_compare(attn, x, 1.0 / math.sqrt(128), True, gpu, f"pairs Hq={Hq} Hkv={Hkv} S={S}")


def test_mqa_and_mha(attn, gpu):
    for Hq, Hkv in ((8, 1), (3, 3)):
        x = make_prefill_inputs(1, Hq, Hkv, 200, 128, seed=30 + Hq)
        full_compare(attn, x, 0.09, True, gpu, f"Hq={Hq} Hkv={Hkv}")


@pytest.mark.parametrize("d", [128, 256])
def test_large_scores_running_max_jumps(attn, gpu, d):
    """Keys scaled so the running max jumps by far more than the lazy-rescale threshold."""
    x = make_prefill_inputs(1, 2, 1, 700, d, seed=44)
    k = x.k.clone()
    k[:, 129::97] *= 8
    k[:, 400:] *= 2
    x.k = k
    full_compare(attn, x, 1.0 / math.sqrt(d), True, gpu, f"max jumps d={d}")


@pytest.mark.parametrize("d", [64, 128, 256])
def test_score_jump_past_the_reference_range(attn, gpu, d):
    """A few keys past the first key tile scaled by 64: against the first tile's row max their
    exponentials would overflow, so every row that sees them must take the row max again and
    rescale (the step's second pass), and rows that do not see them keep the first reference."""
    x = make_prefill_inputs(1, 2, 1, 600, d, seed=45)
    k = x.k.clone()
    k[:, 200::131] *= 64
    x.k = k
    full_compare(attn, x, 1.0 / math.sqrt(d), True, gpu, f"score jump d={d}")
    full_compare(attn, x, 1.0 / math.sqrt(d), False, gpu, f"score jump non-causal d={d}")


@pytest.mark.parametrize("d", [128, 256])
def test_row0_returns_v0_exactly(attn, gpu, d):
    """Causal row 0 sees only key 0, so O[0] = v0 bit-exactly and LSE[0] = scale * q0.k0."""
    x = make_prefill_inputs(2, 4, 2, 130, d, seed=5)
    o, lse = run_prefill(attn, x, 0.1, True, gpu)
    o = o.cpu()
    for h in range(4):
        assert torch.equal(o[:, 0, h], x.v[:, 0, h // 2]), "row 0 must equal v0"


def test_outputs_stay_in_bounds(attn, gpu):
    """Writes stay inside o / lse: guard regions filled with NaN remain NaN."""
    B, S, Hq, Hkv, d = 1, 200, 2, 1, 128
    x = make_prefill_inputs(B, Hq, Hkv, S, d, seed=6)
    q, k, v = (t.to(gpu) for t in (x.q, x.k, x.v))
    n = B * S * Hq * d
    big = torch.full((n + 4096,), float("nan"), dtype=torch.bfloat16, device=gpu)
    o = big[:n].view(B, S, Hq, d)
    lbig = torch.full((B * Hq * S + 1024,), float("nan"), dtype=torch.float32, device=gpu)
    lse = lbig[:B * Hq * S].view(B, Hq, S)
    attn.prefill(q, k, v, scale=0.1, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.isnan(big[n:]).all() and torch.isnan(lbig[B * Hq * S:]).all()
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


def test_deterministic_and_stream(attn, gpu):
    x = make_prefill_inputs(1, 4, 1, 384, 128, seed=7)
    q, k, v = (t.to(gpu) for t in (x.q, x.k, x.v))
    o1, l1 = attn.prefill(q, k, v, scale=0.08)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o2, l2 = attn.prefill(q, k, v, scale=0.08, stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_lse_optional(attn, gpu):
    x = make_prefill_inputs(1, 2, 2, 64, 64, seed=8)
    q, k, v = (t.to(gpu) for t in (x.q, x.k, x.v))
    o, lse = attn.prefill(q, k, v, scale=0.125, return_lse=False)
    torch.cuda.synchronize()
    assert lse is None
    wo, _ = oa.prefill(x.q, x.k, x.v, 0.125)
    check_o(to_np(o), wo, "no lse")


def _sampled(attn, gpu, cfg, heads, nrows, seed):
    """Full-size config, sampled rows (first, last, tile edges, random) of a few heads."""
    x = prefill_inputs_for(cfg)
    o, lse = run_prefill(attn, x, cfg.scale, True, gpu)
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, 256, cfg.S - 129, cfg.S - 1],
                                     rng.integers(0, cfg.S, nrows)]))
    on, ln = to_np(o), to_np(lse)
    for b in range(cfg.B):
        wo, wl = oa.prefill(x.q, x.k, x.v, cfg.scale, causal=True, heads=heads, rows=rows, batches=[b])
        for h in heads:
            check_o(on[b, rows, h], wo[b, rows, h], f"{cfg.name} b={b} h={h}")
            check_lse(ln[b, h, rows], wl[b, h, rows], f"{cfg.name} b={b} h={h}")
    assert np.isfinite(on).all() and np.isfinite(ln).all()


def _complete(attn, gpu, cfg):
    """Full-size config: every output row of every head and batch element against the oracle."""
    x = prefill_inputs_for(cfg)
    o, lse = run_prefill(attn, x, cfg.scale, True, gpu)
    wo, wl = oa.prefill(x.q, x.k, x.v, cfg.scale, causal=True)
    on, ln = to_np(o), to_np(lse)
    for b in range(cfg.B):
        for h in range(cfg.Hq):
            check_o(on[b, :, h], wo[b, :, h], f"{cfg.name} b={b} h={h}")
            check_lse(ln[b, h], wl[b, h], f"{cfg.name} b={b} h={h}")
    check_o(on, wo, f"{cfg.name} all heads")


def test_llama8b_full_size_complete(attn, gpu):
    _complete(attn, gpu, LLAMA8B)


@pytest.mark.parametrize("cfg", [c for c in SWEEP if c.S <= 2048], ids=lambda c: c.name)
def test_sweep_full_size_complete(attn, gpu, cfg):
    _complete(attn, gpu, cfg)


@pytest.mark.parametrize("cfg", [c for c in SWEEP if c.S > 2048], ids=lambda c: c.name)
def test_sweep_full_size_sampled(attn, gpu, cfg):
    _sampled(attn, gpu, cfg, heads=[0, 1, 13, 30, 31], nrows=32, seed=cfg.seed)


def test_d256_8k_prompt_sampled(attn, gpu):
    """Head dim 256 (64-key tiles): Hq=16, Hkv=2, S=8192, scale 2^-4; sampled rows of three heads."""
    _sampled(attn, gpu, QWEN256, heads=[0, 7, 15], nrows=24, seed=9)


def test_vanishing_scale_gives_prefix_means(attn, gpu):
    """scale -> 0 (1e-30; 0 itself is refused): every visible key weighs the same, so row i is the
    mean of v_0..v_i and LSE = ln(i+1)."""
    x = make_prefill_inputs(1, 2, 1, 300, 128, seed=12)
    o, lse = run_prefill(attn, x, 1e-30, True, gpu)
    v = x.v[0, :, 0].double()
    want = torch.cumsum(v, 0) / torch.arange(1, 301, dtype=torch.float64)[:, None]
    for h in range(2):
        check_o(to_np(o)[0, :, h], want.numpy(), "prefix means")
        check_lse(to_np(lse)[0, h], np.log(np.arange(1, 301)), "ln(i+1)")


def test_long_sequence_sampled(attn, gpu):
    """One 32K-token sequence (256 query tiles, up to 256 key tiles per row); sampled rows."""
    cfg_S = 32768
    x = make_prefill_inputs(1, 2, 1, cfg_S, 128, seed=13)
    o, lse = run_prefill(attn, x, 1.0 / math.sqrt(128), True, gpu)
    rows = np.array([0, 1, 127, 128, 4095, 4096, 20000, cfg_S - 129, cfg_S - 1])
    wo, wl = oa.prefill(x.q, x.k, x.v, 1.0 / math.sqrt(128), causal=True, rows=rows)
    check_o(to_np(o)[0, rows], wo[0, rows], "32K rows")
    check_lse(to_np(lse)[0][:, rows], wl[0][:, rows], "32K lse")
