"""The C-ABI library loads and exports everything include/attn.h declares (no GPU needed).

Host-side argument checks run before any CUDA call, so they are exercised here too.
"""
import ctypes

import pytest


def test_exports_every_declared_symbol(attn):
    declared = attn.header_functions()
    assert {"attn_prefill", "attn_decode_paged", "attn_combine"} <= set(declared)
    lib = attn.lib()
    missing = [name for name in declared if not hasattr(lib, name)]
    assert not missing, missing


def test_status_strings(attn):
    lib = attn.lib()
    names = [lib.attn_status_string(i).decode() for i in range(7)]
    assert names[:6] == ["ATTN_OK", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED", "ATTN_ERR_WORKSPACE",
                         "ATTN_ERR_CUDA", "ATTN_ERR_DEVICE"]
    assert names[6] == "ATTN_ERR_UNKNOWN"
    assert lib.attn_version() >= 100


FAKE = 0x10000  # an aligned non-null address; never dereferenced by the host checks below


@pytest.mark.parametrize("args,want", [
    ((None, FAKE, FAKE, FAKE, None, 1, 4, 2, 64, 128, 0.1, 1, None), 1),          # null q
    ((FAKE + 2, FAKE, FAKE, FAKE, None, 1, 4, 2, 64, 128, 0.1, 1, None), 1),      # misaligned q
    ((FAKE, FAKE, FAKE, FAKE, None, 0, 4, 2, 64, 128, 0.1, 1, None), 1),          # B = 0
    ((FAKE, FAKE, FAKE, FAKE, None, 1, 4, 3, 64, 128, 0.1, 1, None), 1),          # Hq % Hkv != 0
    ((FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 0, 128, 0.1, 1, None), 1),           # S = 0
    ((FAKE, FAKE, FAKE, FAKE, FAKE + 1, 1, 4, 2, 64, 128, 0.1, 1, None), 1),      # misaligned lse
    ((FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 64, 96, 0.1, 1, None), 2),           # d = 96 unsupported
    ((FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 64, 128, float("nan"), 1, None), 1), # NaN scale
    ((FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 64, 128, 0.0, 1, None), 1),          # scale 0
    ((FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 64, 128, -0.1, 1, None), 1),         # negative scale
])
def test_prefill_argument_checks(attn, args, want):
    assert attn.lib().attn_prefill(*args) == want


def _decode_args(**over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, lens=FAKE, o=FAKE, lse=None, N=2, Hq=8, Hkv=2, d=128, page=16,
             maxb=4, nblocks=8, ns=2, st=0, scale=0.1, ws=FAKE, wsb=1 << 20, stream=None)
    a.update(over)
    return tuple(a.values())


@pytest.mark.parametrize("over,want", [
    (dict(q=None), 1), (dict(bt=FAKE + 2), 1), (dict(N=0), 1), (dict(Hkv=3), 1),
    (dict(page=32), 2), (dict(d=64), 2), (dict(Hq=40, Hkv=2), 2),
    (dict(ns=-1), 1), (dict(st=24), 1),                      # bad split count; split_tokens not a page multiple
    (dict(scale=0.0), 1), (dict(scale=-1.0), 1),
    (dict(ws=None), 3), (dict(wsb=10), 3), (dict(ws=FAKE + 4), 3),
])
def test_decode_argument_checks(attn, over, want):
    assert attn.lib().attn_decode_paged(*_decode_args(**over)) == want


def _varlen_args(**over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, cu=FAKE, N=3, maxs=100, T=300, Hq=4, Hkv=2, d=128,
             scale=0.1, causal=1, stream=None)
    a.update(over)
    return tuple(a.values())


@pytest.mark.parametrize("over,want", [
    (dict(cu=None), 1), (dict(cu=FAKE + 2), 1), (dict(N=0), 1), (dict(maxs=0), 1), (dict(T=0), 1),
    (dict(Hkv=3), 1), (dict(d=96), 2), (dict(q=FAKE + 8), 1), (dict(scale=float("inf")), 1),
])
def test_prefill_varlen_argument_checks(attn, over, want):
    assert attn.lib().attn_prefill_varlen(*_varlen_args(**over)) == want


def _paged_prefill_args(**over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, cu=FAKE, lens=FAKE, o=FAKE, lse=None, N=2, maxq=64, T=100, Hq=8,
             Hkv=2, d=128, page=16, maxb=8, nblocks=16, scale=0.1, causal=1, stream=None)
    a.update(over)
    return tuple(a.values())


@pytest.mark.parametrize("over,want", [
    (dict(bt=None), 1), (dict(cu=None), 1), (dict(lens=None), 1), (dict(k=None), 1), (dict(v=FAKE + 2), 1),
    (dict(bt=FAKE + 2), 1), (dict(N=0), 1), (dict(maxq=0), 1), (dict(nblocks=0), 1), (dict(maxb=0), 1),
    (dict(page=32), 2), (dict(d=96), 2), (dict(Hkv=3), 1),
])
def test_prefill_paged_argument_checks(attn, over, want):
    assert attn.lib().attn_prefill_paged(*_paged_prefill_args(**over)) == want


def _host_prefill_args(**over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, S=1000, Hq=8, Hkv=2, d=128, scale=0.1, causal=1, chunks=4,
             ws=FAKE, wsb=1 << 30, stream=None)
    a.update(over)
    return tuple(a.values())


@pytest.mark.parametrize("over,want", [
    (dict(q=None), 1), (dict(k=None), 1), (dict(o=None), 1), (dict(ws=None), 1), (dict(ws=FAKE + 16), 1),
    (dict(S=0), 1), (dict(Hkv=3), 1), (dict(Hq=0), 1), (dict(d=96), 2), (dict(chunks=0), 1), (dict(chunks=65), 1),
    (dict(scale=0.0), 1), (dict(scale=float("nan")), 1), (dict(wsb=1000), 3),
])
def test_prefill_host_argument_checks(attn, over, want):
    """Every argument error returns before a CUDA call (so before the copy streams exist)."""
    assert attn.lib().attn_prefill_host(*_host_prefill_args(**over)) == want


def test_prefill_host_workspace_bytes(attn):
    """q, k, v (padded to whole 16-token pages), o, LSE, the block table and the chunk offsets, each
    region rounded up to 256 bytes."""
    S, Hq, Hkv, d = 1000, 8, 2, 128
    up = lambda x: (x + 255) // 256 * 256
    pages = (S + 15) // 16
    want = (2 * up(S * Hq * d * 2) + 2 * up(pages * 16 * Hkv * d * 2) + up(S * Hq * 4) + up(pages * 4)
            + up(64 * 16))
    assert attn.prefill_host_workspace_bytes(S, Hq, Hkv, d, 4) == want
    assert attn.prefill_host_workspace_bytes(S, Hq, Hkv, d, 64) == want   # the offsets take a fixed 64 slots
    assert attn.prefill_host_workspace_bytes(S, Hq, Hkv, d, 0) == 0
    assert attn.prefill_host_workspace_bytes(S, Hq, 3, d, 4) == 0
    assert attn.prefill_host_workspace_bytes(S, Hq, Hkv, 96, 4) == 0


def test_combine_argument_checks(attn):
    lib = attn.lib()
    assert lib.attn_combine(None, FAKE, FAKE, 4, 2, 128, FAKE, None, None) == 1
    assert lib.attn_combine(FAKE, FAKE, FAKE, 0, 2, 128, FAKE, None, None) == 1
    assert lib.attn_combine(FAKE, FAKE, FAKE, 4, 2, 100, FAKE, None, None) == 2


def test_split_slots_and_workspace(attn):
    assert attn.decode_num_slots(512, num_splits=16) == 16
    assert attn.decode_num_slots(3, num_splits=16) == 3          # never more groups than pages
    assert attn.decode_num_slots(7680, split_tokens=512) == 240
    assert attn.decode_num_slots(10, split_tokens=24) == 0        # not a page multiple
    assert attn.decode_workspace_bytes(64, 32, 128, 1) == 0
    assert attn.decode_workspace_bytes(64, 32, 128, 16) == 64 * 32 * 16 * 130 * 4


def test_binding_refuses_without_library(attn, monkeypatch, tmp_path):
    import attention_attn_prefill_gb300._lib as L
    monkeypatch.setattr(L, "_lib", None)
    monkeypatch.setattr(L, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        L.lib()
