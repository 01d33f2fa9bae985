"""Paged split-KV decode and combine parity against the float64 oracle (through the C ABI)."""
import math

import numpy as np
import pytest
import torch

import oracle.attention as oa
from parity import check_lse, check_o, to_np
from workloads import LONGCTX, PAGED, decode_inputs_for, make_decode_inputs
from workloads.teaching import teaching_scores_values

pytestmark = pytest.mark.gpu


def run_decode(attn, x, scale, dev, **kw):
    args = [t.to(dev) for t in (x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens)]
    o, lse = attn.decode_paged(*args, scale=scale, **kw)
    torch.cuda.synchronize()
    return o, lse


def compare(attn, x, scale, dev, what, seqs=None, **kw):
    o, lse = run_decode(attn, x, scale, dev, **kw)
    wo, wl = oa.decode_paged(x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens, scale, seqs=seqs)
    sel = list(range(x.q.shape[0])) if seqs is None else list(seqs)
    check_o(to_np(o)[sel], wo[sel], what)
    check_lse(to_np(lse)[sel], wl[sel], what)
    return o, lse


@pytest.mark.parametrize("kw", [dict(num_splits=1), dict(num_splits=4), dict(num_splits=16),
                                dict(num_splits=3), dict(split_tokens=16), dict(split_tokens=48),
                                dict(num_splits=0)],
                         ids=lambda k: "-".join(f"{a}{b}" for a, b in k.items()))
def test_paged_d128_gqa4(attn, gpu, kw):
    """Ragged lengths (1..700), NaN in unused page tails and in unused pages."""
    lens = [1, 15, 16, 17, 31, 64, 100, 129, 255, 256, 257, 500, 700]
    x = make_decode_inputs(lens, Hq=32, Hkv=8, d=128, seed=51, nan_tail=True, extra_blocks=5)
    compare(attn, x, 1.0 / math.sqrt(128), gpu, f"d128 {kw}", **kw)


@pytest.mark.parametrize("kw", [dict(num_splits=1), dict(num_splits=5), dict(split_tokens=64),
                                dict(split_tokens=512), dict(num_splits=0)],
                         ids=lambda k: "-".join(f"{a}{b}" for a, b in k.items()))
def test_paged_d256_gqa8(attn, gpu, kw):
    lens = [1, 33, 200, 513, 1000, 1300]
    x = make_decode_inputs(lens, Hq=16, Hkv=2, d=256, seed=52, nan_tail=True, extra_blocks=3)
    compare(attn, x, 2.0 ** -4, gpu, f"d256 {kw}", **kw)


@pytest.mark.parametrize("hq_hkv", [(1, 1), (16, 1), (6, 3)])
def test_group_sizes(attn, gpu, hq_hkv):
    Hq, Hkv = hq_hkv
    x = make_decode_inputs([40, 77, 300], Hq=Hq, Hkv=Hkv, d=128, seed=53)
    compare(attn, x, 0.1, gpu, f"G={Hq // Hkv}", num_splits=2)


def test_empty_sequence(attn, gpu):
    """seq_len 0 gives o = 0 and lse = -inf; its neighbours are unaffected."""
    lens = [0, 20, 0, 33]
    x = make_decode_inputs(lens, Hq=4, Hkv=1, d=128, seed=54)
    for kw in (dict(num_splits=1), dict(num_splits=4), dict(num_splits=0)):
        o, lse = run_decode(attn, x, 0.1, gpu, **kw)
        o, lse = o.cpu(), lse.cpu()
        assert torch.all(o[[0, 2]] == 0) and torch.all(torch.isneginf(lse[[0, 2]]))
        wo, wl = oa.decode_paged(x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens, 0.1, seqs=[1, 3])
        check_o(to_np(o)[[1, 3]], wo[[1, 3]], f"neighbours {kw}")
        check_lse(to_np(lse)[[1, 3]], wl[[1, 3]], f"neighbours {kw}")


def test_single_token_returns_value(attn, gpu):
    x = make_decode_inputs([1, 1], Hq=8, Hkv=2, d=128, seed=55)
    o, lse = run_decode(attn, x, 0.3, gpu, num_splits=1)
    o = o.cpu()
    for n in range(2):
        pid = int(x.block_table[n, 0])
        for h in range(8):
            assert torch.equal(o[n, h], x.v_cache[pid, 0, h // 4])


def test_split_counts_agree(attn, gpu):
    """Different split geometries agree within the bf16 tolerance (not bit-exactly)."""
    x = make_decode_inputs([3000, 1234, 4096], Hq=32, Hkv=8, d=128, seed=56)
    outs = [run_decode(attn, x, 0.09, gpu, **kw) for kw in (dict(num_splits=1), dict(num_splits=16),
                                                           dict(split_tokens=256), dict(num_splits=0))]
    for o, lse in outs[1:]:
        check_o(to_np(o), to_np(outs[0][0]), "split vs unsplit")
        check_lse(to_np(lse), to_np(outs[0][1]), "split vs unsplit")


def test_balanced_many_short_sequences(attn, gpu):
    """Balanced mode with fewer pages than worker warps (idle warps) and many empty sequences."""
    lens = [0, 1, 0, 0, 17, 3, 0, 16, 40] * 5
    x = make_decode_inputs(lens, Hq=8, Hkv=2, d=128, seed=59, nan_tail=True)
    seqs = [i for i, L in enumerate(lens) if L > 0]
    compare(attn, x, 0.1, gpu, "balanced short", seqs=seqs, num_splits=0)
    o, lse = run_decode(attn, x, 0.1, gpu, num_splits=0)
    empty = [i for i, L in enumerate(lens) if L == 0]
    assert torch.all(o.cpu()[empty] == 0) and torch.all(torch.isneginf(lse.cpu()[empty]))


def test_auto_split_count(attn, gpu):
    """num_splits="auto": the split-count rule for this device, then the usual parity."""
    lens = [3000, 17, 1234, 4096, 640]
    x = make_decode_inputs(lens, Hq=32, Hkv=8, d=128, seed=60, nan_tail=True)
    n = attn.decode_auto_splits(len(lens), 8, 128, x.block_table.shape[1])
    assert 1 <= n <= 128
    compare(attn, x, 0.09, gpu, f"auto ({n} splits)", num_splits="auto")


def test_auto_split_tokens(attn, gpu):
    """split_tokens="auto": the length-aware group size for this device, then the usual parity."""
    lens = [3000, 17, 1234, 9000, 640, 0, 5000]
    x = make_decode_inputs(lens, Hq=16, Hkv=2, d=256, seed=61, nan_tail=True)
    t = attn.decode_auto_split_tokens(x.seq_lens, 2, 256, x.block_table.shape[1])
    assert t >= 16 and t % 16 == 0
    live = [n for n, L in enumerate(lens) if L > 0]
    compare(attn, x, 2.0 ** -4, gpu, f"auto ({t}-token groups)", seqs=live, split_tokens="auto")


@pytest.mark.parametrize("seed", range(6))
def test_random_shapes_and_split_modes(attn, gpu, seed):
    """Seeded random batches (empty, one-token and long sequences; 1 to 8 query heads per KV head;
    d = 128 or 256) under a random split choice; every non-empty sequence against the oracle."""
    rng = np.random.default_rng(1000 + seed)
    N = int(rng.integers(1, 24))
    lens = [int(v) for v in rng.choice([0, 1, 15, 16, 17, 300, 1000, 2500, 5000], size=N)]
    lens[int(rng.integers(0, N))] = int(rng.integers(1, 6000))
    Hq, Hkv = [(8, 1), (16, 2), (12, 4), (32, 8), (6, 6)][int(rng.integers(0, 5))]
    d = [128, 256][int(rng.integers(0, 2))]
    x = make_decode_inputs(lens, Hq=Hq, Hkv=Hkv, d=d, seed=2000 + seed, nan_tail=True, extra_blocks=2)
    modes = [dict(num_splits=int(rng.integers(1, 21))), dict(split_tokens=int(rng.choice([16, 48, 512, 1024]))),
             dict(num_splits=0), dict(split_tokens="auto")]
    kw = modes[seed % len(modes)]
    live = [n for n, L in enumerate(lens) if L > 0]
    if not live:
        return
    compare(attn, x, float(d) ** -0.5, gpu, f"seed {seed} N={N} G={Hq // Hkv} d={d} {kw}", seqs=live, **kw)


def test_bad_page_is_reported(attn, gpu):
    """A block-table entry outside [0, num_blocks) is recorded as a device error, not read."""
    x = make_decode_inputs([40], Hq=4, Hkv=1, d=128, seed=57)
    bt = x.block_table.clone()
    bt[0, 1] = x.num_blocks + 1000
    args = [t.to(gpu) for t in (x.q, x.k_cache, x.v_cache, bt, x.seq_lens)]
    attn.decode_paged(*args, scale=0.1, num_splits=1)
    assert attn.device_status(clear=True) == 2


def test_worked_example_on_gpu(attn, gpu):
    """The 27,525-token teaching input: one-hot query, k_t = score_t e_0, v_t = value_t.

    The exact output is 1.325056137248; the bf16 result must be one of its two
    bf16 neighbours, 1.3203125 or 1.328125 ("Plugging in actual numbers").
    """
    s, v = teaching_scores_values()
    L, d = len(s), 128
    x = make_decode_inputs([L], Hq=1, Hkv=1, d=d, seed=58)
    x.q.zero_()
    x.q[0, 0, 0] = 1.0
    kc = torch.zeros_like(x.k_cache)
    vc = torch.zeros_like(x.v_cache)
    pids = x.block_table[0].tolist()
    st = torch.tensor(s, dtype=torch.bfloat16)
    vt = torch.tensor(v, dtype=torch.bfloat16)
    assert torch.equal(st.double(), torch.tensor(s, dtype=torch.float64))   # exact in bf16
    for p, pid in enumerate(pids):
        a, b = 16 * p, min(16 * p + 16, L)
        kc[pid, :b - a, 0, 0] = st[a:b]
        vc[pid, :b - a, 0, :] = vt[a:b, None]
    x.k_cache, x.v_cache = kc, vc
    for kw in (dict(num_splits=1), dict(num_splits=54), dict(split_tokens=448), dict(split_tokens=320),
               dict(num_splits=0)):
        o, lse = run_decode(attn, x, 1.0, gpu, **kw)
        vals = set(o[0, 0].float().cpu().tolist())
        assert len(vals) == 1 and vals.pop() in (1.3203125, 1.328125), kw


_FULL = {}


def _full_size(cfg):
    """The config's inputs and the oracle's output for every sequence, computed once per session."""
    if cfg.name not in _FULL:
        x = decode_inputs_for(cfg)
        _FULL[cfg.name] = (x, oa.decode_paged(x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens, cfg.scale))
    return _FULL[cfg.name]


def _compare_full(attn, cfg, dev, what, **kw):
    x, (wo, wl) = _full_size(cfg)
    o, lse = run_decode(attn, x, cfg.scale, dev, **kw)
    check_o(to_np(o), wo, what)
    check_lse(to_np(lse), wl, what)


@pytest.mark.parametrize("kw", [dict(num_splits=n) for n in PAGED.num_splits] + [dict(num_splits=0), dict(auto=1)],
                         ids=lambda k: "-".join(f"{a}{b}" for a, b in k.items()))
def test_paged_config_full_size(attn, gpu, kw):
    """64 sequences, lengths U[512, 8192], GQA 32:8, d=128: every output of every sequence, per split
    choice (num_splits 0 is balanced mode; auto is the length-aware group size)."""
    if "auto" in kw:
        x, _ = _full_size(PAGED)
        kw = dict(split_tokens=attn.decode_auto_split_tokens(x.seq_lens, PAGED.Hkv, PAGED.d, x.block_table.shape[1]))
    _compare_full(attn, PAGED, gpu, f"paged {kw}", **kw)


@pytest.mark.parametrize("span", LONGCTX.split_tokens + (0, "auto"))
def test_longctx_config_full_size(attn, gpu, span):
    """8 sequences up to 122,863 tokens, Hq=16, Hkv=2, d=256, scale 2^-4: every output, per group size.

    span 0 is balanced mode; auto is the length-aware group size."""
    if span == "auto":
        x, _ = _full_size(LONGCTX)
        span = attn.decode_auto_split_tokens(x.seq_lens, LONGCTX.Hkv, LONGCTX.d, x.block_table.shape[1])
    _compare_full(attn, LONGCTX, gpu, f"longctx span={span}", split_tokens=span)


# ------------------------------------------------------------------ combine


@pytest.mark.parametrize("d", [64, 128, 256])
def test_combine_matches_oracle(attn, gpu, d):
    rng = np.random.default_rng(d)
    rows, splits = 37, 9
    po = rng.standard_normal((rows, splits, d)).astype(np.float32)
    pm = (rng.standard_normal((rows, splits)) * 20).astype(np.float32)
    pl = rng.uniform(0.5, 300, (rows, splits)).astype(np.float32)
    empty = rng.random((rows, splits)) < 0.2
    empty[3, :] = False
    pm[empty], pl[empty], po[empty] = -np.inf, 0.0, 0.0
    empty_row = 5
    pm[empty_row], pl[empty_row], po[empty_row] = -np.inf, 0.0, 0.0
    t = lambda a: torch.from_numpy(a).to(gpu)
    o, lse = attn.combine(t(po), t(pm), t(pl))
    torch.cuda.synchronize()
    o, lse = to_np(o), to_np(lse)
    for r in range(rows):
        if r == empty_row:
            assert np.all(o[r] == 0) and np.isneginf(lse[r])
            continue
        wo, wl = oa.combine(po[r].astype(np.float64), pm[r].astype(np.float64), pl[r].astype(np.float64))
        # bf16 rounding of O: half an ulp relative, plus f32 accumulation
        assert np.all(np.abs(o[r] - wo) <= 2.0 ** -8 * np.abs(wo) + 1e-5), r
        assert abs(lse[r] - wl) <= 1e-4 * (1 + abs(wl)), r
