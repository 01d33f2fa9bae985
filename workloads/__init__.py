"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module only draws random numbers and lays them out in the tensor shapes
the attention library consumes. It holds none of the attention arithmetic, so
the CUDA path and the float64 oracle can both be fed from it without sharing
any code that computes a result.

Recipe (the pages give shapes but not a generator):
  * every tensor is drawn on the CPU with ``torch.Generator().manual_seed(seed)``
    as float32 standard normal values and then rounded to bfloat16 (round to
    nearest even), so both machines see bit-identical inputs;
  * the "K scaled by 2 on 1% of rows" sweep picks ceil(0.01*S) token positions
    per batch element with a seeded permutation and doubles every KV head's key
    there (exact in bfloat16: only the exponent changes);
  * paged caches use 16-token pages; the physical pages of all sequences are
    placed by one seeded random permutation, and the block table maps each
    sequence's logical page p to its physical page;
  * the unused tail of each sequence's last page can be filled with NaN so that
    a kernel reading past ``seq_len`` shows up as a NaN in its output.

Shapes follow the library's layouts: prefill q/o ``[B, S, Hq, d]``,
k/v ``[B, S, Hkv, d]``; decode q/o ``[N, Hq, d]``, caches
``[num_blocks, page, Hkv, d]``, block table ``[N, max_blocks]`` int32,
sequence lengths ``[N]`` int32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

PAGE_TOKENS = 16


@dataclass(frozen=True)
class PrefillConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    S: int
    d: int
    scale: float
    seed: int
    k_boost_frac: float = 0.0
    causal: bool = True

    @property
    def causal_flops(self) -> float:
        """Multiply-adds of S = QK^T and O = PV over the visible (query, key) pairs, x2."""
        pairs = self.S * (self.S + 1) / 2 if self.causal else float(self.S) * self.S
        return 4.0 * self.B * self.Hq * self.d * pairs

    @property
    def s2_flops(self) -> float:
        """The same count under the S^2/2 convention for causal pairs (S^2 when not causal)."""
        pairs = self.S * self.S / 2 if self.causal else float(self.S) * self.S
        return 4.0 * self.B * self.Hq * self.d * pairs

    @property
    def min_bytes(self) -> int:
        """Q + K + V + O in bf16 plus the f32 LSE."""
        qo = 2 * self.B * self.S * self.Hq * self.d * 2
        kv = 2 * self.B * self.S * self.Hkv * self.d * 2
        return qo + kv + 4 * self.B * self.Hq * self.S


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    N: int
    Hq: int
    Hkv: int
    d: int
    scale: float
    seed: int
    lens: tuple[int, ...] | None = None     # fixed lengths, else drawn
    len_lo: int = 0
    len_hi: int = 0
    num_splits: tuple[int, ...] = (1,)
    split_tokens: tuple[int, ...] = ()


# The five workloads.  Shapes come from the pages: the Llama-3.1-8B prefill cell
# (GQA 32:8, S=2048, d=128) of "GPU Datapath: Where Every Byte Moves in One LLM
# Inference Step", section C; its paged decode cell (16-token shuffled pages),
# section D; and the Qwen decode of "Why your local LLM feels dumber than it is"
# (d=256, scale 2^-4, context depths from its prompt-depth table).
TINY = PrefillConfig("tiny", B=1, Hq=1, Hkv=1, S=128, d=64, scale=1.0 / 8.0, seed=0)
LLAMA8B = PrefillConfig("llama8b_prefill", B=1, Hq=32, Hkv=8, S=2048, d=128,
                        scale=1.0 / math.sqrt(128.0), seed=1)
SWEEP = tuple(
    PrefillConfig(f"sweep_s{s}", B=4, Hq=32, Hkv=8, S=s, d=128,
                  scale=1.0 / math.sqrt(128.0), seed=seed, k_boost_frac=0.01)
    for s, seed in ((1024, 2), (2048, 3), (4096, 4))
)
PAGED = DecodeConfig("paged_decode", N=64, Hq=32, Hkv=8, d=128,
                     scale=1.0 / math.sqrt(128.0), seed=5, len_lo=512, len_hi=8192,
                     num_splits=(1, 4, 16))
LONGCTX = DecodeConfig("longctx_decode", N=8, Hq=16, Hkv=2, d=256, scale=2.0 ** -4, seed=6,
                       lens=(6335, 19873, 27525, 42192, 67144, 83233, 94146, 122863),
                       split_tokens=(512, 1024, 2048, 4096))

# Extra measurement (not one of the five workloads): the long-context decode model's heads
# (Hq=16, Hkv=2, d=256, scale 2^-4) prefilling an 8K-token prompt.
QWEN256 = PrefillConfig("qwen_d256_prefill", B=1, Hq=16, Hkv=2, S=8192, d=256, scale=2.0 ** -4, seed=7)

PREFILL_CONFIGS = (TINY, LLAMA8B) + SWEEP + (QWEN256,)
DECODE_CONFIGS = (PAGED, LONGCTX)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, gen: torch.Generator) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


@dataclass
class PrefillInputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    boosted_rows: list = field(default_factory=list)


def make_prefill_inputs(B: int, Hq: int, Hkv: int, S: int, d: int, seed: int,
                        k_boost_frac: float = 0.0) -> PrefillInputs:
    g = _gen(seed)
    q = randn_bf16((B, S, Hq, d), g)
    k = randn_bf16((B, S, Hkv, d), g)
    v = randn_bf16((B, S, Hkv, d), g)
    boosted = []
    if k_boost_frac > 0.0:
        n = max(1, math.ceil(k_boost_frac * S))
        for b in range(B):
            rows = torch.randperm(S, generator=g)[:n].sort().values
            k[b, rows] = k[b, rows] * 2          # exact: exponent + 1
            boosted.append(rows.tolist())
    return PrefillInputs(q, k, v, boosted)


def prefill_inputs_for(cfg: PrefillConfig) -> PrefillInputs:
    return make_prefill_inputs(cfg.B, cfg.Hq, cfg.Hkv, cfg.S, cfg.d, cfg.seed, cfg.k_boost_frac)


@dataclass
class VarlenInputs:
    q: torch.Tensor           # [T, Hq, d] bf16, the sequences back to back
    k: torch.Tensor           # [T, Hkv, d] bf16
    v: torch.Tensor
    cu_seqlens: torch.Tensor  # [N + 1] int32 token offsets
    extra: int = 0            # tokens after the last sequence (belong to none)

    @property
    def max_seqlen(self) -> int:
        return int((self.cu_seqlens[1:] - self.cu_seqlens[:-1]).max())


def make_varlen_inputs(lens, Hq: int, Hkv: int, d: int, seed: int, extra: int = 0) -> VarlenInputs:
    """Packed sequences of the given lengths (zero allowed), N(0,1) bf16; ``extra`` trailing tokens
    that belong to no sequence."""
    g = _gen(seed)
    T = int(sum(lens)) + extra
    q = randn_bf16((T, Hq, d), g)
    k = randn_bf16((T, Hkv, d), g)
    v = randn_bf16((T, Hkv, d), g)
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    return VarlenInputs(q, k, v, cu, extra)


@dataclass
class DecodeInputs:
    q: torch.Tensor            # [N, Hq, d] bf16
    k_cache: torch.Tensor      # [num_blocks, PAGE, Hkv, d] bf16
    v_cache: torch.Tensor
    block_table: torch.Tensor  # [N, max_blocks] int32
    seq_lens: torch.Tensor     # [N] int32

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])


def decode_lens_for(cfg: DecodeConfig) -> list[int]:
    if cfg.lens is not None:
        return list(cfg.lens)
    g = _gen(cfg.seed * 1000 + 17)
    return torch.randint(cfg.len_lo, cfg.len_hi + 1, (cfg.N,), generator=g).tolist()


def make_decode_inputs(lens, Hq: int, Hkv: int, d: int, seed: int, *, nan_tail: bool = False,
                       extra_blocks: int = 0, page: int = PAGE_TOKENS) -> DecodeInputs:
    """Paged decode inputs with a shuffled block table.

    ``extra_blocks`` physical pages that no sequence uses are added (filled with
    NaN when ``nan_tail``) so that a stray page index would poison the output.
    """
    lens = [int(x) for x in lens]
    N = len(lens)
    g = _gen(seed)
    pages_per_seq = [(L + page - 1) // page for L in lens]
    used = sum(pages_per_seq)
    num_blocks = used + int(extra_blocks)
    max_blocks = max(1, max(pages_per_seq) if pages_per_seq else 1)
    q = randn_bf16((N, Hq, d), g)
    k_cache = randn_bf16((num_blocks, page, Hkv, d), g)
    v_cache = randn_bf16((num_blocks, page, Hkv, d), g)
    perm = torch.randperm(num_blocks, generator=g)[:used].to(torch.int32)
    block_table = torch.zeros((N, max_blocks), dtype=torch.int32)
    cursor = 0
    for n, npg in enumerate(pages_per_seq):
        block_table[n, :npg] = perm[cursor:cursor + npg]
        cursor += npg
    if nan_tail:
        nan = torch.tensor(float("nan"), dtype=torch.bfloat16)
        for n, L in enumerate(lens):
            npg = pages_per_seq[n]
            if npg and L % page:
                pid = int(block_table[n, npg - 1])
                k_cache[pid, L % page:] = nan
                v_cache[pid, L % page:] = nan
        if extra_blocks:
            mask = torch.ones(num_blocks, dtype=torch.bool)
            mask[perm.long()] = False
            k_cache[mask] = nan
            v_cache[mask] = nan
    return DecodeInputs(q, k_cache, v_cache, block_table, torch.tensor(lens, dtype=torch.int32))


@dataclass
class ChunkedInputs:
    q: torch.Tensor             # [T, Hq, d] bf16: the new tokens of every sequence, back to back
    k_cache: torch.Tensor       # [num_blocks, PAGE, Hkv, d] bf16 (all cached tokens, new ones included)
    v_cache: torch.Tensor
    block_table: torch.Tensor   # [N, max_blocks] int32
    seq_lens: torch.Tensor      # [N] int32 cached tokens per sequence
    cu_seqlens_q: torch.Tensor  # [N + 1] int32 offsets of the new tokens

    @property
    def max_seqlen_q(self) -> int:
        return max(1, int((self.cu_seqlens_q[1:] - self.cu_seqlens_q[:-1]).max()))


def make_chunked_inputs(ctx_lens, q_lens, Hq: int, Hkv: int, d: int, seed: int, **kw) -> ChunkedInputs:
    """A paged cache of ctx_lens tokens per sequence (as make_decode_inputs) and q_lens new query
    tokens per sequence (its last q_lens cached tokens), packed."""
    if any(int(a) > int(b) for a, b in zip(q_lens, ctx_lens)):
        raise ValueError("a chunk cannot be longer than its sequence")
    x = make_decode_inputs(ctx_lens, Hq, Hkv, d, seed, **kw)
    g = _gen(seed + 7919)
    q = randn_bf16((int(sum(q_lens)), Hq, d), g)
    cu = torch.zeros(len(q_lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor([int(v) for v in q_lens], dtype=torch.int64), 0).to(torch.int32)
    return ChunkedInputs(q, x.k_cache, x.v_cache, x.block_table, x.seq_lens, cu)


def decode_inputs_for(cfg: DecodeConfig, **kw) -> DecodeInputs:
    return make_decode_inputs(decode_lens_for(cfg), cfg.Hq, cfg.Hkv, cfg.d, cfg.seed, **kw)


def decode_kv_bytes(lens, Hkv: int, d: int) -> int:
    """K and V bytes one decode step must read (bf16)."""
    return int(sum(lens)) * Hkv * d * 2 * 2


def decode_min_bytes(lens, Hq: int, Hkv: int, d: int, page: int = PAGE_TOKENS,
                     with_lse: bool = True) -> int:
    """Algorithmic bytes of one decode step: K+V, q, o, (lse), block-table entries, lens."""
    N = len(lens)
    kv = decode_kv_bytes(lens, Hkv, d)
    qo = 2 * N * Hq * d * 2
    lse = 4 * N * Hq if with_lse else 0
    bt = 4 * sum((int(L) + page - 1) // page for L in lens)
    return kv + qo + lse + bt + 4 * N


@dataclass
class PartialInputs:
    part_o: torch.Tensor  # [rows, splits, d] f32: a group's stored value
    part_m: torch.Tensor  # [rows, splits] f32: group max (-inf where empty)
    part_l: torch.Tensor  # [rows, splits] f32: group sum of weights (0 where empty)


def make_partials(rows: int, splits: int, d: int, seed: int, *, empty_frac: float = 0.2,
                  empty_rows=(), m_spread: float = 3.0) -> PartialInputs:
    """Random per-group partials for merge tests: m ~ N(0, m_spread), l ~ U[1, 300), the stored
    values N(0, 1) times a per-group magnitude in [1, 50); slots are empty with probability
    ``empty_frac`` (every slot of the rows in ``empty_rows``)."""
    g = _gen(seed)
    m = torch.randn((rows, splits), generator=g) * m_spread
    l = 1.0 + 299.0 * torch.rand((rows, splits), generator=g)
    mag = 1.0 + 49.0 * torch.rand((rows, splits, 1), generator=g)
    o = torch.randn((rows, splits, d), generator=g) * mag
    empty = torch.rand((rows, splits), generator=g) < empty_frac
    for r in empty_rows:
        empty[r] = True
    m[empty] = float("-inf")
    l[empty] = 0.0
    o[empty] = 0.0
    return PartialInputs(o.float().contiguous(), m.float().contiguous(), l.float().contiguous())
