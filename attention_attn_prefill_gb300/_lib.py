"""ctypes binding of libattn.so: argument marshalling only.

Every computation happens in the library's CUDA kernels; these wrappers only
check tensor shapes/dtypes, allocate outputs (and the decode workspace) with
torch, and pass raw device pointers plus the current CUDA stream.  If the
library is missing they raise -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import math
import os
import re

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libattn.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "attn.h")

_STATUS = {
    0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_WORKSPACE",
    4: "ATTN_ERR_CUDA", 5: "ATTN_ERR_DEVICE",
}
PAGE_TOKENS = 16


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {_STATUS.get(status, status)}")
        self.status = status


_lib = None

c_int, c_float, c_void_p, c_size_t = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
c_u32_p = ctypes.POINTER(ctypes.c_uint32)

_SIGNATURES = {
    "attn_status_string": (ctypes.c_char_p, [c_int]),
    "attn_version": (c_int, []),
    "attn_prefill": (c_int, [c_void_p] * 5 + [c_int] * 5 + [c_float, c_int, c_void_p]),
    "attn_decode_num_slots": (c_int, [c_int] * 4),
    "attn_decode_workspace_bytes": (c_size_t, [c_int] * 4),
    "attn_decode_balanced_workspace_bytes": (c_size_t, [c_int] * 4),
    "attn_decode_paged": (c_int, [c_void_p] * 7 + [c_int] * 9 + [c_float, c_void_p, c_size_t, c_void_p]),
    "attn_combine": (c_int, [c_void_p] * 3 + [c_int] * 3 + [c_void_p, c_void_p, c_void_p]),
    "attn_decode_paged_noalloc": (c_int, [c_void_p] * 7 + [c_int] * 9 + [c_float, c_void_p]),
    "attn_device_status": (c_int, [c_u32_p, c_int]),
    "attn_split_heuristic": (c_int, [c_int] * 4),
    "attn_prefill_varlen": (c_int, [c_void_p] * 6 + [c_int] * 6 + [c_float, c_int, c_void_p]),
    "attn_prefill_paged": (c_int, [c_void_p] * 8 + [c_int] * 9 + [c_float, c_int, c_void_p]),
    "attn_prefill_host": (c_int, [c_void_p] * 5 + [c_int] * 4 + [c_float, c_int, c_int, c_void_p, c_size_t, c_void_p]),
    "attn_prefill_host_workspace_bytes": (c_size_t, [c_int] * 5),
    "attn_decode_auto_splits": (c_int, [c_int] * 4),
    "attn_split_tokens_rule": (c_int, [c_void_p] + [c_int] * 4),
    "attn_decode_auto_split_tokens": (c_int, [c_void_p] + [c_int] * 4),
    "attn_emulated_partitions": (c_int, [c_int] * 5),
    "attn_emulated_num_slots": (c_int, [c_int] * 4),
    "attn_emulated_workspace_bytes": (c_size_t, [c_int] * 4),
    "attn_decode_paged_emulated": (c_int, [c_void_p] * 7 + [c_int] * 9 + [c_float, c_void_p, c_size_t, c_void_p]),
    "attn_merge_emulated": (c_int, [c_int] + [c_void_p] * 3 + [c_int] * 3 + [c_void_p] * 4),
}

# Decode numerics of other backends (attn_numerics_t).
NUMERICS = {"triton": 1, "fa2": 2, "xqa": 3, "trt": 4}


def library_path() -> str:
    return LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded libattn.so (loaded once).  Raises if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with attention_attn_prefill_gb300.build.build()")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def header_functions() -> list[str]:
    """Names of the entry points include/attn.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


def _check(status: int, where: str) -> None:
    if status != 0:
        raise AttnError(status, where)


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream or 0)


def _dev(t: torch.Tensor, dtype, name: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def prefill(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float | None = None, causal: bool = True,
            out: torch.Tensor | None = None, lse: torch.Tensor | None = None, return_lse: bool = True,
            stream=None):
    """Prefill attention: q [B,S,Hq,d], k/v [B,S,Hkv,d] bf16 -> (o [B,S,Hq,d] bf16, lse [B,Hq,S] f32)."""
    B, S, Hq, d = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, S, Hkv, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, S, Hkv, d] matching q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    st = lib().attn_prefill(
        _dev(q, torch.bfloat16, "q"), _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"),
        _dev(out, torch.bfloat16, "out"), _dev(lse, torch.float32, "lse") if lse is not None else None,
        B, Hq, Hkv, S, d, float(scale), 1 if causal else 0, _stream_handle(stream))
    _check(st, "attn_prefill")
    return out, lse


def prefill_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens: torch.Tensor, max_seqlen: int,
                   scale: float | None = None, causal: bool = True, out: torch.Tensor | None = None,
                   lse: torch.Tensor | None = None, return_lse: bool = True, stream=None):
    """Packed sequences: q [T,Hq,d], k/v [T,Hkv,d] bf16, cu_seqlens [N+1] int32 -> (o [T,Hq,d], lse [Hq,T])."""
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (T, Hkv, d) or v.shape != k.shape:
        raise ValueError("k and v must be [total_tokens, Hkv, d] matching q")
    if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
        raise ValueError("cu_seqlens must be [num_seqs + 1]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device)
    st = lib().attn_prefill_varlen(
        _dev(q, torch.bfloat16, "q"), _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"),
        _dev(out, torch.bfloat16, "out"), _dev(lse, torch.float32, "lse") if lse is not None else None,
        _dev(cu_seqlens, torch.int32, "cu_seqlens"), cu_seqlens.numel() - 1, int(max_seqlen), T, Hq, Hkv, d,
        float(scale), 1 if causal else 0, _stream_handle(stream))
    _check(st, "attn_prefill_varlen")
    return out, lse


def prefill_paged(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: torch.Tensor,
                  cu_seqlens_q: torch.Tensor, seq_lens: torch.Tensor, max_seqlen_q: int, scale: float | None = None,
                  causal: bool = True, out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                  return_lse: bool = True, stream=None):
    """Chunked prefill: new tokens q [T,Hq,d] against the paged cache [num_blocks,16,Hkv,d] -> (o, lse [Hq,T])."""
    T, Hq, d = q.shape
    num_blocks, page, Hkv, dk = k_cache.shape
    if dk != d or v_cache.shape != k_cache.shape:
        raise ValueError("caches must be [num_blocks, page, Hkv, d] matching q")
    N = seq_lens.numel()
    if block_table.dim() != 2 or block_table.shape[0] != N or cu_seqlens_q.shape != (N + 1,):
        raise ValueError("block_table must be [N, max_blocks], cu_seqlens_q [N+1] and seq_lens [N]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device)
    st = lib().attn_prefill_paged(
        _dev(q, torch.bfloat16, "q"), _dev(k_cache, torch.bfloat16, "k_cache"),
        _dev(v_cache, torch.bfloat16, "v_cache"), _dev(block_table, torch.int32, "block_table"),
        _dev(cu_seqlens_q, torch.int32, "cu_seqlens_q"), _dev(seq_lens, torch.int32, "seq_lens"),
        _dev(out, torch.bfloat16, "out"), _dev(lse, torch.float32, "lse") if lse is not None else None,
        N, int(max_seqlen_q), T, Hq, Hkv, d, page, block_table.shape[1], num_blocks, float(scale),
        1 if causal else 0, _stream_handle(stream))
    _check(st, "attn_prefill_paged")
    return out, lse


def _host(t: torch.Tensor, dtype, name: str) -> int:
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def prefill_host_workspace_bytes(S: int, Hq: int, Hkv: int, d: int, chunks: int = 4) -> int:
    return int(lib().attn_prefill_host_workspace_bytes(S, Hq, Hkv, d, chunks))


def prefill_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float | None = None, causal: bool = True,
                 chunks: int = 4, out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                 return_lse: bool = True, workspace: torch.Tensor | None = None, device=None, stream=None):
    """Prefill of one sequence in host memory: q [S,Hq,d], k/v [S,Hkv,d] bf16 (pinned for overlap) ->
    (o [S,Hq,d] bf16, lse [Hq,S] f32) in host memory, complete once `stream` reaches the call's end.
    The transfers overlap the compute inside the call (attn_prefill_host); `workspace` is a device
    uint8 tensor of prefill_host_workspace_bytes(...) bytes (allocated on `device` if not given)."""
    S, Hq, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (S, Hkv, d) or v.shape != k.shape:
        raise ValueError("k and v must be [S, Hkv, d] matching q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    pin = q.is_pinned()
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=pin)
    if lse is None and return_lse:
        lse = torch.empty((Hq, S), dtype=torch.float32, pin_memory=pin)
    need = prefill_host_workspace_bytes(S, Hq, Hkv, d, chunks)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8,
                                device=device if device is not None else torch.device("cuda", torch.cuda.current_device()))
    st = lib().attn_prefill_host(
        _host(q, torch.bfloat16, "q"), _host(k, torch.bfloat16, "k"), _host(v, torch.bfloat16, "v"),
        _host(out, torch.bfloat16, "out"), _host(lse, torch.float32, "lse") if lse is not None else None,
        S, Hq, Hkv, d, float(scale), 1 if causal else 0, int(chunks), _dev(workspace, torch.uint8, "workspace"),
        workspace.numel(), _stream_handle(stream))
    _check(st, "attn_prefill_host")
    return out, lse


def decode_num_slots(max_blocks_per_seq: int, num_splits: int = 1, split_tokens: int = 0,
                     page_size: int = PAGE_TOKENS) -> int:
    return int(lib().attn_decode_num_slots(max_blocks_per_seq, page_size, num_splits, split_tokens))


def decode_workspace_bytes(num_seqs: int, Hq: int, d: int, slots: int) -> int:
    return int(lib().attn_decode_workspace_bytes(num_seqs, Hq, d, slots))


def split_heuristic(units: int, capacity: int, blocks: int, max_splits: int = 128) -> int:
    """The split-count rule restated in C (host arithmetic only); 0 for invalid arguments."""
    return int(lib().attn_split_heuristic(units, capacity, blocks, max_splits))


def decode_auto_splits(num_seqs: int, Hkv: int, d: int, max_blocks_per_seq: int) -> int:
    """Split count the rule picks for the split kernel on the current device."""
    n = int(lib().attn_decode_auto_splits(num_seqs, Hkv, d, max_blocks_per_seq))
    if n < 1:
        raise AttnError(1, "attn_decode_auto_splits")
    return n


def _host_lens(seq_lens) -> tuple[ctypes.Array, int]:
    vals = [int(x) for x in (seq_lens.tolist() if isinstance(seq_lens, torch.Tensor) else seq_lens)]
    return (ctypes.c_int32 * max(1, len(vals)))(*vals), len(vals)


def split_tokens_rule(seq_lens, Hkv: int, capacity: int, max_blocks_per_seq: int) -> int:
    """Length-aware group size (host arithmetic only) for given host lengths; 0 for invalid arguments."""
    arr, n = _host_lens(seq_lens)
    return int(lib().attn_split_tokens_rule(ctypes.addressof(arr), n, Hkv, capacity, max_blocks_per_seq))


def decode_auto_split_tokens(seq_lens, Hkv: int, d: int, max_blocks_per_seq: int) -> int:
    """split_tokens the length-aware rule picks on the current device, from host lengths."""
    arr, n = _host_lens(seq_lens)
    t = int(lib().attn_decode_auto_split_tokens(ctypes.addressof(arr), n, Hkv, d, max_blocks_per_seq))
    if t < 1:
        raise AttnError(1, "attn_decode_auto_split_tokens")
    return t


def decode_balanced_workspace_bytes(num_seqs: int, Hq: int, Hkv: int, d: int) -> int:
    return int(lib().attn_decode_balanced_workspace_bytes(num_seqs, Hq, Hkv, d))


def decode_paged(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: torch.Tensor,
                 seq_lens: torch.Tensor, scale: float | None = None, num_splits: int = 1, split_tokens: int = 0,
                 out: torch.Tensor | None = None, lse: torch.Tensor | None = None, return_lse: bool = True,
                 workspace: torch.Tensor | None = None, stream=None):
    """Paged split-KV decode: q [N,Hq,d]; caches [num_blocks,16,Hkv,d] bf16 -> (o [N,Hq,d], lse [N,Hq]).

    num_splits=0 with split_tokens=0 selects balanced mode (equal page shares per worker warp);
    num_splits="auto" takes the count decode_auto_splits picks; split_tokens="auto" takes the group
    size decode_auto_split_tokens picks from the lengths (read back to the host once, a device sync).
    """
    N, Hq, d = q.shape
    num_blocks, page, Hkv, dk = k_cache.shape
    if dk != d or v_cache.shape != k_cache.shape:
        raise ValueError("caches must be [num_blocks, page, Hkv, d] matching q")
    if block_table.dim() != 2 or block_table.shape[0] != N or seq_lens.shape != (N,):
        raise ValueError("block_table must be [N, max_blocks] and seq_lens [N]")
    max_blocks = block_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if num_splits == "auto":
        num_splits = decode_auto_splits(N, Hkv, d, max_blocks)
    if split_tokens == "auto":
        split_tokens = decode_auto_split_tokens(seq_lens.cpu(), Hkv, d, max_blocks)
        num_splits = 0
    if num_splits == 0 and split_tokens == 0:
        need = int(lib().attn_decode_balanced_workspace_bytes(N, Hq, Hkv, d))   # balanced mode
        if need == 0:
            raise AttnError(1, "attn_decode_balanced_workspace_bytes")
    else:
        slots = decode_num_slots(max_blocks, num_splits, split_tokens, page)
        if slots < 1:
            raise AttnError(1, "attn_decode_num_slots")
        need = decode_workspace_bytes(N, Hq, d, slots)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((N, Hq), dtype=torch.float32, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().attn_decode_paged(
        _dev(q, torch.bfloat16, "q"), _dev(k_cache, torch.bfloat16, "k_cache"),
        _dev(v_cache, torch.bfloat16, "v_cache"), _dev(block_table, torch.int32, "block_table"),
        _dev(seq_lens, torch.int32, "seq_lens"), _dev(out, torch.bfloat16, "out"),
        _dev(lse, torch.float32, "lse") if lse is not None else None,
        N, Hq, Hkv, d, page, max_blocks, num_blocks, num_splits, split_tokens, float(scale), ws_ptr, ws_bytes,
        _stream_handle(stream))
    _check(st, "attn_decode_paged")
    return out, lse


def decode_paged_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: torch.Tensor,
                         seq_lens: torch.Tensor, scale: float | None = None, num_splits: int = 1,
                         split_tokens: int = 0, out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                         return_lse: bool = True, stream=None):
    """decode_paged without a workspace: the partials use the library's fixed device array."""
    N, Hq, d = q.shape
    num_blocks, page, Hkv, _ = k_cache.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((N, Hq), dtype=torch.float32, device=q.device)
    st = lib().attn_decode_paged_noalloc(
        _dev(q, torch.bfloat16, "q"), _dev(k_cache, torch.bfloat16, "k_cache"),
        _dev(v_cache, torch.bfloat16, "v_cache"), _dev(block_table, torch.int32, "block_table"),
        _dev(seq_lens, torch.int32, "seq_lens"), _dev(out, torch.bfloat16, "out"),
        _dev(lse, torch.float32, "lse") if lse is not None else None,
        N, Hq, Hkv, d, page, block_table.shape[1], num_blocks, num_splits, split_tokens, float(scale),
        _stream_handle(stream))
    _check(st, "attn_decode_paged_noalloc")
    return out, lse


def combine(part_o: torch.Tensor, part_m: torch.Tensor, part_l: torch.Tensor, out: torch.Tensor | None = None,
            lse: torch.Tensor | None = None, return_lse: bool = True, stream=None):
    """Merge partials: part_o [rows, splits, d], part_m/part_l [rows, splits] f32 -> (o [rows,d] bf16, lse [rows])."""
    rows, splits, d = part_o.shape
    if part_m.shape != (rows, splits) or part_l.shape != (rows, splits):
        raise ValueError("part_m and part_l must be [rows, splits]")
    if out is None:
        out = torch.empty((rows, d), dtype=torch.bfloat16, device=part_o.device)
    if lse is None and return_lse:
        lse = torch.empty((rows,), dtype=torch.float32, device=part_o.device)
    st = lib().attn_combine(
        _dev(part_o, torch.float32, "part_o"), _dev(part_m, torch.float32, "part_m"),
        _dev(part_l, torch.float32, "part_l"), rows, splits, d, _dev(out, torch.bfloat16, "out"),
        _dev(lse, torch.float32, "lse") if lse is not None else None, _stream_handle(stream))
    _check(st, "attn_combine")
    return out, lse


def _numerics(name: str) -> int:
    if name not in NUMERICS:
        raise ValueError(f"numerics must be one of {sorted(NUMERICS)}")
    return NUMERICS[name]


def emulated_partitions(numerics: str, num_seqs: int, Hkv: int, max_tokens: int, sm_count: int) -> int:
    """Group count the backend would pick on a GPU of ``sm_count`` SMs (host arithmetic only)."""
    n = int(lib().attn_emulated_partitions(_numerics(numerics), num_seqs, Hkv, max_tokens, sm_count))
    if n < 1:
        raise AttnError(1, "attn_emulated_partitions")
    return n


def emulated_num_slots(numerics: str, max_blocks_per_seq: int, partitions: int = 0,
                       page_size: int = PAGE_TOKENS) -> int:
    return int(lib().attn_emulated_num_slots(_numerics(numerics), max_blocks_per_seq, page_size, partitions))


def decode_paged_emulated(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: torch.Tensor,
                          seq_lens: torch.Tensor, numerics: str, partitions: int | None = None,
                          sm_count: int | None = None, max_tokens: int | None = None, scale: float | None = None,
                          out: torch.Tensor | None = None, lse: torch.Tensor | None = None, return_lse: bool = True,
                          workspace: torch.Tensor | None = None, stream=None):
    """Paged decode with another backend's numerics ("triton", "fa2", "xqa" or "trt").

    ``partitions`` defaults to the count the backend picks for ``max_tokens`` (the block table's
    capacity if not given) on a GPU of ``sm_count`` SMs (this device's if not given).  Returns
    (o, lse, workspace); the workspace holds the per-group partials (see include/attn.h).
    """
    N, Hq, d = q.shape
    num_blocks, page, Hkv, dk = k_cache.shape
    if dk != d or v_cache.shape != k_cache.shape:
        raise ValueError("caches must be [num_blocks, page, Hkv, d] matching q")
    if block_table.dim() != 2 or block_table.shape[0] != N or seq_lens.shape != (N,):
        raise ValueError("block_table must be [N, max_blocks] and seq_lens [N]")
    max_blocks = block_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if partitions is None:
        if sm_count is None:
            sm_count = torch.cuda.get_device_properties(q.device).multi_processor_count
        partitions = emulated_partitions(numerics, N, Hkv, max_tokens or max_blocks * page, sm_count)
    slots = emulated_num_slots(numerics, max_blocks, partitions, page)
    if slots < 1:
        raise AttnError(1, "attn_emulated_num_slots")
    need = int(lib().attn_emulated_workspace_bytes(N, Hq, d, slots))
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((N, Hq), dtype=torch.float32, device=q.device)
    st = lib().attn_decode_paged_emulated(
        _dev(q, torch.bfloat16, "q"), _dev(k_cache, torch.bfloat16, "k_cache"),
        _dev(v_cache, torch.bfloat16, "v_cache"), _dev(block_table, torch.int32, "block_table"),
        _dev(seq_lens, torch.int32, "seq_lens"), _dev(out, torch.bfloat16, "out"),
        _dev(lse, torch.float32, "lse") if lse is not None else None,
        N, Hq, Hkv, d, page, max_blocks, num_blocks, _numerics(numerics), partitions, float(scale),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(st, "attn_decode_paged_emulated")
    return out, lse, workspace


def emulated_partials(workspace: torch.Tensor, N: int, Hq: int, d: int, slots: int):
    """Views of the partials a call of decode_paged_emulated left in its workspace:
    (part_o [N*Hq, slots, d], part_m [N*Hq, slots], part_l [N*Hq, slots])."""
    f = workspace.view(torch.float32)
    rows = N * Hq
    po = f[:rows * slots * d].view(rows, slots, d)
    pm = f[rows * slots * d:rows * slots * (d + 1)].view(rows, slots)
    pl = f[rows * slots * (d + 1):rows * slots * (d + 2)].view(rows, slots)
    return po, pm, pl


def merge_emulated(numerics: str, part_o: torch.Tensor, part_m: torch.Tensor, part_l: torch.Tensor,
                   want_f32: bool = True, want_bf16: bool = True, return_lse: bool = True, stream=None):
    """A backend's merge on given partials: part_o [rows, splits, d], part_m/part_l [rows, splits] f32
    -> (o_f32 [rows, d] or None, o [rows, d] bf16 or None, lse [rows] or None)."""
    rows, splits, d = part_o.shape
    if part_m.shape != (rows, splits) or part_l.shape != (rows, splits):
        raise ValueError("part_m and part_l must be [rows, splits]")
    dev = part_o.device
    o32 = torch.empty((rows, d), dtype=torch.float32, device=dev) if want_f32 else None
    o = torch.empty((rows, d), dtype=torch.bfloat16, device=dev) if want_bf16 else None
    lse = torch.empty((rows,), dtype=torch.float32, device=dev) if return_lse else None
    st = lib().attn_merge_emulated(
        _numerics(numerics), _dev(part_o, torch.float32, "part_o"), _dev(part_m, torch.float32, "part_m"),
        _dev(part_l, torch.float32, "part_l"), rows, splits, d,
        _dev(o32, torch.float32, "o_f32") if o32 is not None else None,
        _dev(o, torch.bfloat16, "o") if o is not None else None,
        _dev(lse, torch.float32, "lse") if lse is not None else None, _stream_handle(stream))
    _check(st, "attn_merge_emulated")
    return o32, o, lse


def device_status(clear: bool = True) -> int:
    """First device-side error code recorded by a kernel (0 = none); synchronises the device."""
    code = ctypes.c_uint32(0)
    _check(lib().attn_device_status(ctypes.byref(code), 1 if clear else 0), "attn_device_status")
    return int(code.value)
