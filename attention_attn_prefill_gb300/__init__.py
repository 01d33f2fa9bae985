"""GB300-native exact attention: causal prefill, paged split-KV decode, LSE combine.

The compute lives in ``libattn.so`` (hand-written sm_103a CUDA behind the C
ABI of ``include/attn.h``); this package is its Python binding.
"""
from ._lib import (NUMERICS, AttnError, combine, decode_auto_split_tokens, decode_auto_splits,
                   decode_balanced_workspace_bytes,
                   decode_num_slots, decode_paged, decode_paged_emulated, decode_paged_noalloc,
                   decode_workspace_bytes, device_status, emulated_num_slots, emulated_partials,
                   emulated_partitions, header_functions, lib, library_path, merge_emulated, prefill, prefill_host,
                   prefill_host_workspace_bytes, prefill_paged, prefill_varlen, split_heuristic, split_tokens_rule)

__all__ = [
    "NUMERICS", "AttnError", "combine", "decode_auto_split_tokens", "decode_auto_splits", "decode_balanced_workspace_bytes", "decode_num_slots",
    "decode_paged", "decode_paged_emulated", "decode_paged_noalloc", "decode_workspace_bytes", "device_status",
    "emulated_num_slots", "emulated_partials", "emulated_partitions", "header_functions", "lib", "library_path",
    "merge_emulated", "prefill", "prefill_host", "prefill_host_workspace_bytes", "prefill_paged", "prefill_varlen", "split_heuristic", "split_tokens_rule",
]
