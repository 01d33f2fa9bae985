"""A wait that runs out ends the kernel with an error status; the GPU stays usable.

Every mbarrier wait in the kernels gives up after ATTN_WAIT_LIMIT_NS and records device status 1
(kDevWaitTimeout); the warp that gave up waits (again with a limit) for its own copies in flight
and still reaches every CTA barrier, so the kernel ends.  That path is exercised here on the paged
decode's split kernel through a test-only build of the library, compiled with a 2 ms limit and
ATTN_TEST_DROP_COPY: with the hook switched on, one warp of one CTA never requests its first page,
so the wait for that page runs out.  Nothing faults, traps or hangs: the only failure is a
barrier that nothing completes.  The test checks that the call returns promptly, that the status
reads 1, and that the next call on the same device is correct again.
"""
import ctypes
import math
import time

import numpy as np
import pytest
import torch

import oracle.attention as oa
from parity import check_lse, check_o, to_np
from workloads import make_decode_inputs

pytestmark = pytest.mark.gpu

WAIT_LIMIT_NS = 2_000_000   # the test build's limit: 2 ms


@pytest.fixture(scope="module")
def waittest_lib():
    from attention_attn_prefill_gb300.build import build
    path = build(variant="waittest", extra_flags=["-DATTN_TEST_DROP_COPY", f"-DATTN_WAIT_LIMIT_NS={WAIT_LIMIT_NS}ull"])
    lib = ctypes.CDLL(path)
    vp, ci, cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.attn_decode_paged.restype = ci
    lib.attn_decode_paged.argtypes = [vp] * 7 + [ci] * 9 + [cf, vp, ctypes.c_size_t, vp]
    lib.attn_device_status.restype = ci
    lib.attn_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), ci]
    lib.attn_test_drop_copy.restype = ci
    lib.attn_test_drop_copy.argtypes = [ci]
    return lib


def _decode(lib, x, scale, dev):
    q, kc, vc, bt, sl = (t.to(dev) for t in (x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens))
    N, Hq, d = q.shape
    num_blocks, page, Hkv, _ = kc.shape
    o = torch.full_like(q, float("nan"))
    lse = torch.full((N, Hq), float("nan"), dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st = lib.attn_decode_paged(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), sl.data_ptr(), o.data_ptr(),
                               lse.data_ptr(), N, Hq, Hkv, d, page, bt.shape[1], num_blocks, 1, 0, scale, None, 0,
                               torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return st, o, lse, time.perf_counter() - t0


def _status(lib):
    code = ctypes.c_uint32(0)
    assert lib.attn_device_status(ctypes.byref(code), 1) == 0
    return int(code.value)


def test_wait_that_runs_out_ends_with_status_and_device_recovers(waittest_lib, gpu):
    lib = waittest_lib
    x = make_decode_inputs([700, 1500, 90], Hq=8, Hkv=2, d=128, seed=81, nan_tail=True)
    scale = 1.0 / math.sqrt(128)
    assert _status(lib) == 0

    assert lib.attn_test_drop_copy(1) == 0
    st, o, _, seconds = _decode(lib, x, scale, gpu)
    assert st == 0                      # the launch itself is fine; the error is recorded on the device
    assert _status(lib) == 1            # kDevWaitTimeout
    # two waits run out (the consumer's and the drain's), each after the 2 ms limit; nothing hangs
    assert seconds < 2.0, seconds
    # the sequences no warp of CTA (0, 0, 0) serves are unaffected
    wo, wl = oa.decode_paged(x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens, scale)
    check_o(to_np(o)[1:], wo[1:], "unaffected sequences after a timed-out wait")

    # the device and the library are usable again, and correct
    assert lib.attn_test_drop_copy(0) == 0
    st, o, lse, _ = _decode(lib, x, scale, gpu)
    assert st == 0 and _status(lib) == 0
    check_o(to_np(o), wo, "decode after recovery")
    check_lse(to_np(lse), wl, "decode after recovery")
    assert torch.isfinite(torch.ones(4, device=gpu).sum())
