"""The bounded mbarrier wait that every kernel of the library uses.

A test-only kernel (tests/csrc/wait_probe.cu, its own library over the
kernels' common.cuh) waits on an mbarrier that nothing arrives on, with no
copy in flight and a short limit: the wait must give up, the kernel must
return and record PKV_DEVERR_TIMEOUT, and the context must stay usable.  The
same kernel with one arrival must pass the wait at once with no error.
"""
import ctypes

import pytest
import torch

from paged_kv_cache_41_gb300 import build as pkv_build
from paged_kv_cache_41_gb300 import pkv

pytestmark = pytest.mark.gpu


def _probe():
    lib = ctypes.CDLL(pkv_build.build_wait_probe())
    fn = lib.pkv_test_wait_probe
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.POINTER(ctypes.c_uint),
                   ctypes.POINTER(ctypes.c_ulonglong)]

    def run(limit_ns, arrive):
        err, el = ctypes.c_uint(0xFFFFFFFF), ctypes.c_ulonglong(0)
        rc = fn(limit_ns, arrive, ctypes.byref(err), ctypes.byref(el))
        assert rc == 0, f"cuda error {rc}"
        return err.value, el.value
    return run


def test_wait_that_nobody_completes_times_out_and_reports():
    torch.cuda.init()
    run = _probe()
    limit = 2_000_000  # 2 ms
    err, elapsed = run(limit, 0)
    assert err == pkv.DEVERR_TIMEOUT
    assert limit <= elapsed < 1_000_000_000
    # the context is still usable: a completed wait passes with no error
    err, elapsed = run(limit, 1)
    assert err == 0 and elapsed < limit
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float(x.sum()) == 1023 * 1024 / 2
