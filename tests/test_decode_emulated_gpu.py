"""Paged decode with other backends' numerics against the oracle (through the C ABI).

"Why your local LLM feels dumber than it is" (Part 3.14), section "Backend names expand into four
decode algorithms".  Three levels:
  * the merge kernel on given partials is bit-identical to the oracle's float32 merges
    (each operation rounded on its own, exp / log rounded once from double);
  * each group partial the split kernel leaves in the workspace matches the float64 partial of the
    oracle's group of tokens for that backend (this checks the geometry: contiguous 16-token tiles,
    64-token blocks, round-robin 256-token tiles, 128-token tiles) and has the backend's stored type;
  * the merged output equals exact attention within the decode tolerance, at small and full size.
"""
import math

import numpy as np
import pytest
import torch

import oracle.attention as oa
import oracle.split_sim as ss
from oracle import numerics as nx
from parity import LSE_ABS, check_lse, check_o, to_np
from workloads import LONGCTX, PAGED, decode_inputs_for, make_decode_inputs, make_partials
from workloads.teaching import teaching_scores_values

pytestmark = pytest.mark.gpu

BACKENDS = ss.BACKENDS


def check_backend_lse(backend, got, want, what=""):
    """XQA's sum of weights adds bf16-rounded weights (relative rounding at most 2^-9 each), so its
    log-sum-exp may be off by up to 2^-9 on top of the usual bound; the other backends sum float32
    weights and keep the usual bound."""
    if backend != "xqa":
        return check_lse(got, want, what or backend)
    err = np.abs(np.asarray(got, np.float64) - np.asarray(want, np.float64))
    assert err.max() <= LSE_ABS + 2.0 ** -9, f"{what or backend}: lse max abs err {err.max():.4g}"


def _bits(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32)).view(np.uint32)


# ------------------------------------------------------------------ merge kernel, bit for bit

@pytest.mark.parametrize("backend", BACKENDS)
@pytest.mark.parametrize("d,splits", [(64, 1), (128, 5), (128, 200), (256, 300), (1000, 7), (3, 600)])
def test_merge_bit_exact(attn, gpu, backend, d, splits):
    """Register prefetch (few groups, other d) and shared-memory staging (96 or more groups at d of
    128 or 256) both keep the slot order: bit-identical results either way."""
    rows = 6
    x = make_partials(rows, splits, d, seed=1000 + d + splits, empty_frac=0.25, empty_rows=(2,))
    o32, o, lse = attn.merge_emulated(backend, x.part_o.to(gpu), x.part_m.to(gpu), x.part_l.to(gpu))
    torch.cuda.synchronize()
    o32, o, lse = o32.cpu().numpy(), o.float().cpu().numpy(), lse.cpu().numpy()
    po, pm, pl = x.part_o.numpy(), x.part_m.numpy(), x.part_l.numpy()
    for r in range(rows):
        live = pl[r] > 0
        if not live.any():
            assert not o32[r].any() and not o[r].any() and lse[r] == -np.inf
            continue
        want, want_lse = ss.merge(backend, po[r][live], pm[r][live], pl[r][live])
        assert np.array_equal(_bits(o32[r]), _bits(want)), f"row {r}: f32 result differs"
        assert np.array_equal(_bits(o[r]), _bits(nx.bf16_array(want))), f"row {r}: bf16 result differs"
        assert _bits(lse[r]) == _bits(want_lse), f"row {r}: lse {lse[r]!r} vs {float(want_lse)!r}"


def test_merge_teaching_groups_bit_exact(attn, gpu):
    """The page's 27,525-token example: the oracle's float32 groups of every backend, merged on the GPU."""
    s, v = teaching_scores_values()
    for backend in BACKENDS:
        for sm in (132, 148, 188):
            L = len(s)
            parts_n = {"fa2": ss.fa2_split_count(L, sm)[0], "xqa": ss.xqa_partition_count(L, sm)}.get(backend, 16)
            groups = ss.backend_groups(backend, L, parts_n)
            st = [ss.group_partial(s, v, g, **ss.GROUP_OPTIONS[backend]) for g in groups]
            stored = [p.weighted_sum if ss.STORED[backend] == "numerator" else p.normalised_output for p in st]
            po = torch.tensor(stored, dtype=torch.float32).view(1, -1, 1)
            pm = torch.tensor([p.local_max for p in st], dtype=torch.float32).view(1, -1)
            pl = torch.tensor([p.norm_sum for p in st], dtype=torch.float32).view(1, -1)
            o32, o, _ = attn.merge_emulated(backend, po.to(gpu), pm.to(gpu), pl.to(gpu))
            want = ss.simulate(backend, s, v, sm)
            assert float(o32.item()) == want.f32_output, (backend, sm)
            assert float(o.float().item()) == want.bf16_output, (backend, sm)


# ------------------------------------------------------------------ split kernel partials

class _OracleGroups:
    """Float64 partials (o, m, l) of a backend's groups, per (sequence, query head)."""

    def __init__(self, x, scale):
        self.x, self.scale = x, scale
        self.kc, self.vc, self.q = oa.f64(x.k_cache), oa.f64(x.v_cache), oa.f64(x.q)
        self.Hq, self.Hkv = x.q.shape[1], x.k_cache.shape[2]
        self._seq = {}

    def __call__(self, backend, partitions, n, hq):
        L = int(self.x.seq_lens[n])
        if n not in self._seq:
            bt = self.x.block_table[n].numpy()
            self._seq[n] = (oa.gather_pages(self.kc, bt, L, 16), oa.gather_pages(self.vc, bt, L, 16))
        keys, vals = self._seq[n]
        g = oa.kv_head_of(hq, self.Hq, self.Hkv)
        return [oa.partial(self.q[n, hq], keys[idx, g], vals[idx, g], self.scale)
                for idx in (ss.backend_groups(backend, L, partitions) if L else [])]


@pytest.mark.parametrize("backend", BACKENDS)
@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("partitions", [1, 3, 16])
def test_partials_and_output(attn, gpu, backend, d, partitions):
    if backend == "trt" and partitions != 3:
        pytest.skip("TensorRT-LLM's groups do not depend on a count")
    lens = [0, 1, 15, 16, 17, 255, 256, 257, 700, 1500, 3001]
    Hq, Hkv = (8, 2) if d == 128 else (16, 2)
    scale = 1.0 / math.sqrt(d)
    x = make_decode_inputs(lens, Hq=Hq, Hkv=Hkv, d=d, seed=70 + d, nan_tail=True, extra_blocks=3)
    args = [t.to(gpu) for t in (x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens)]
    o, lse, ws = attn.decode_paged_emulated(*args, numerics=backend, partitions=partitions, scale=scale)
    torch.cuda.synchronize()
    slots = attn.emulated_num_slots(backend, x.max_blocks, partitions)
    po, pm, pl = (to_np(t) for t in attn.emulated_partials(ws, len(lens), Hq, d, slots))
    bf16_stored = backend in ("xqa", "trt")
    groups_of = _OracleGroups(x, scale)
    for n, L in enumerate(lens):
        for hq in range(0, Hq, 3):
            row = n * Hq + hq
            want = groups_of(backend, partitions, n, hq)
            assert len(want) <= slots
            for s in range(slots):
                if s >= len(want):
                    assert pm[row, s] == -np.inf and pl[row, s] == 0 and not po[row, s].any(), (n, hq, s)
                    continue
                wo, wm, wl = want[s]
                what = f"{backend} n={n} L={L} hq={hq} group {s}"
                assert abs(pm[row, s] - wm) < 1e-3, what
                assert abs(pl[row, s] / wl - 1) < 5e-3, (what, pl[row, s], wl)
                stored = po[row, s]
                if bf16_stored:
                    assert np.array_equal(stored, nx.bf16_array(stored.astype(np.float32))), what
                got = stored / pl[row, s] if ss.STORED[backend] == "numerator" else stored
                check_o(got, wo, what)
    wo, wl = oa.decode_paged(x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens, scale)
    live = [n for n, L in enumerate(lens) if L > 0]
    check_o(to_np(o)[live], wo[live], backend)
    check_backend_lse(backend, to_np(lse)[live], wl[live])
    empty = [n for n, L in enumerate(lens) if L == 0]
    assert not to_np(o)[empty].any() and np.all(to_np(lse)[empty] == -np.inf)


@pytest.mark.parametrize("backend", BACKENDS)
@pytest.mark.parametrize("hq_hkv,d", [((16, 1), 128), ((4, 4), 256), ((32, 2), 128)])
def test_group_shapes_and_more_groups_than_tiles(attn, gpu, backend, hq_hkv, d):
    """All 16 MMA rows in use (G = 16), one query head per KV head (G = 1), and G = 16 at d = 128 with
    two KV heads; 40 groups, more than the short sequences have tiles; wide CTAs (a small grid) and
    the default shape (40 groups x sequences x KV heads above the SM count) both run."""
    Hq, Hkv = hq_hkv
    lens = [3, 100, 600, 2500, 5000]
    x = make_decode_inputs(lens, Hq=Hq, Hkv=Hkv, d=d, seed=80 + Hq + d, nan_tail=True)
    args = [t.to(gpu) for t in (x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens)]
    scale = 1.0 / math.sqrt(d)
    for parts in (40, 2):
        o, lse, _ = attn.decode_paged_emulated(*args, numerics=backend, partitions=parts, scale=scale)
        torch.cuda.synchronize()
        wo, wl = oa.decode_paged(x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens, scale)
        check_o(to_np(o), wo, f"{backend} G={Hq // Hkv} d={d} parts={parts}")
        check_backend_lse(backend, to_np(lse), wl, f"{backend} G={Hq // Hkv} parts={parts}")


def test_worked_example_every_backend(attn, gpu):
    """The teaching input (one-hot query, k_t = score_t e_0, v_t = value_t) through each backend's
    geometry for H200, B200 and SM120: every result is one of the two bf16 neighbours of the exact
    1.325056137248 ("Plugging in actual numbers")."""
    s, v = teaching_scores_values()
    L, d = len(s), 128
    x = make_decode_inputs([L], Hq=1, Hkv=1, d=d, seed=58)
    x.q.zero_()
    x.q[0, 0, 0] = 1.0
    kc = torch.zeros_like(x.k_cache)
    vc = torch.zeros_like(x.v_cache)
    st = torch.tensor(s, dtype=torch.bfloat16)
    vt = torch.tensor(v, dtype=torch.bfloat16)
    for p, pid in enumerate(x.block_table[0].tolist()):
        a, b = 16 * p, min(16 * p + 16, L)
        kc[pid, :b - a, 0, 0] = st[a:b]
        vc[pid, :b - a, 0, :] = vt[a:b, None]
    args = [t.to(gpu) for t in (x.q, kc, vc, x.block_table, x.seq_lens)]
    for backend in BACKENDS:
        for sm in (132, 148, 188):
            o, _, _ = attn.decode_paged_emulated(*args, numerics=backend, sm_count=sm, max_tokens=L, scale=1.0)
            vals = set(o[0, 0].float().cpu().tolist())
            assert len(vals) == 1 and vals.pop() in (1.3203125, 1.328125), (backend, sm)


# ------------------------------------------------------------------ full size

@pytest.fixture(scope="module")
def longctx():
    x = decode_inputs_for(LONGCTX)
    return x, oa.decode_paged(x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens, LONGCTX.scale)


@pytest.fixture(scope="module")
def paged():
    x = decode_inputs_for(PAGED)
    return x, oa.decode_paged(x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens, PAGED.scale)


@pytest.mark.parametrize("backend", BACKENDS)
def test_longctx_full_size(attn, gpu, backend, longctx):
    """8 sequences up to 122,863 tokens, d = 256, each backend's B200 (148 SMs) group count; every output."""
    x, (wo, wl) = longctx
    args = [t.to(gpu) for t in (x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens)]
    o, lse, _ = attn.decode_paged_emulated(*args, numerics=backend, sm_count=148, scale=LONGCTX.scale,
                                           max_tokens=int(x.seq_lens.max()))
    torch.cuda.synchronize()
    check_o(to_np(o), wo, f"longctx {backend}")
    check_backend_lse(backend, to_np(lse), wl, f"longctx {backend}")


@pytest.mark.parametrize("backend", BACKENDS)
def test_paged_full_size(attn, gpu, backend, paged):
    """64 sequences of U[512, 8192] tokens, GQA 32:8, d = 128, this GPU's group counts; every output."""
    x, (wo, wl) = paged
    args = [t.to(gpu) for t in (x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens)]
    o, lse, _ = attn.decode_paged_emulated(*args, numerics=backend, scale=PAGED.scale,
                                           max_tokens=int(x.seq_lens.max()))
    torch.cuda.synchronize()
    check_o(to_np(o), wo, f"paged {backend}")
    check_backend_lse(backend, to_np(lse), wl, f"paged {backend}")
