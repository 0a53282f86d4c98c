"""The allocation-free decode entry point against the regular one.

pkv_paged_attention_decode_static serves callers that may not allocate device
memory (a host framework that owns every allocation, or a steady-state serving
loop that must never call cudaMalloc/cudaFree).  Its split-K scratch is a fixed
array the library declares in device memory and shares between calls.  This
test calls it three times in a row through the C ABI, on different batches, and
checks each result against pkv_paged_attention_decode with a caller-owned
workspace, within the attention tolerance |a - b| <= 2e-3 + 1e-2 |b|.  It also
checks that sizes beyond the array are refused.  The file is named to be
collected last.
"""
import gc

import numpy as np
import pytest
import torch

from paged_kv_cache_41_gb300 import pkv
from paged_kv_cache_41_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2


def _pool(b):
    shape = (b.num_blocks, b.block_size, b.num_kv_heads, b.head_dim)
    dt = wl.DTYPES[b.dtype]
    kc = torch.zeros(shape, dtype=dt, device="cuda")
    vc = torch.zeros(shape, dtype=dt, device="cuda")
    slots = torch.from_numpy(b.slots).cuda()
    pkv.kv_append(kc, vc, b.k_hist, b.v_hist, slots)
    return kc, vc


def _close(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    both_inf = np.isinf(b) & (a == b)
    with np.errstate(invalid="ignore"):
        err = np.where(both_inf, 0.0, np.abs(a - b))
    return bool(np.all(err <= ATOL + RTOL * np.where(both_inf, 0.0, np.abs(b))))


def test_static_scratch_matches_workspace_version_on_successive_calls():
    batches = [
        wl.custom_batch([1000, 37, 4096, 0, 513, 2000], dtype="bf16", hq=32, hkv=8, d=128, p=16,
                        seed=71, device="cuda"),
        wl.custom_batch([300, 7000, 64, 1500], dtype="bf16", hq=16, hkv=4, d=128, p=64,
                        seed=72, device="cuda"),
        # eight query heads per kv head: the tensor-core decode
        wl.custom_batch([900, 5, 3000, 129], dtype="bf16", hq=64, hkv=8, d=128, p=16,
                        seed=73, device="cuda"),
    ]
    for b in batches:
        kc, vc = _pool(b)
        bt = torch.from_numpy(b.block_tables).cuda()
        sl = torch.from_numpy(b.seq_lens).cuda()
        lse_ref = torch.empty(b.num_seqs, b.num_q_heads, dtype=torch.float32, device="cuda")
        lse_st = torch.empty_like(lse_ref)
        ref = pkv.paged_attention_decode(b.q, kc, vc, bt, sl, b.scale, lse=lse_ref,
                                         partition_size=256)
        got = pkv.paged_attention_decode_static(b.q, kc, vc, bt, sl, b.scale, lse=lse_st,
                                                partition_size=256)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        assert _close(got, ref) and _close(lse_st, lse_ref)


def test_static_scratch_refuses_oversized_requests():
    kc = torch.zeros(8, 16, 8, 128, dtype=torch.bfloat16, device="cuda")
    b, hq, max_blocks = 512, 32, 4096
    need = pkv.decode_workspace_bytes(kc, b, hq, max_blocks, 256)
    assert need > pkv.STATIC_SCRATCH_BYTES
    q = torch.zeros(b, hq, 128, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(b, max_blocks, dtype=torch.int32, device="cuda")
    sl = torch.ones(b, dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.PkvError) as ei:
        pkv.paged_attention_decode_static(q, kc, kc, bt, sl, 1.0, partition_size=256)
    assert ei.value.status == pkv.PKV_ERR_CAPACITY


def test_static_calls_allocate_no_device_memory():
    # out and lse are the caller's; the first call on the device looks up the
    # scratch array's address (and loads the kernels), so it comes first.
    # After it, several calls must leave both torch's allocator and the
    # device's free memory exactly as they were.
    b = wl.custom_batch([1000, 37, 4096, 0, 513, 2000], dtype="bf16", hq=32, hkv=8, d=128, p=16,
                        seed=74, device="cuda")
    kc, vc = _pool(b)
    bt = torch.from_numpy(b.block_tables).cuda()
    sl = torch.from_numpy(b.seq_lens).cuda()
    out = torch.empty_like(b.q)
    lse = torch.empty(b.num_seqs, b.num_q_heads, dtype=torch.float32, device="cuda")
    ref_lse = torch.empty_like(lse)
    ref = pkv.paged_attention_decode(b.q, kc, vc, bt, sl, b.scale, lse=ref_lse)
    pkv.paged_attention_decode_static(b.q, kc, vc, bt, sl, b.scale, out=out, lse=lse)
    torch.cuda.synchronize()
    # tensors of earlier tests must not be freed by the garbage collector
    # inside the measured calls: that would move the counts the other way
    gc.collect()
    gc.disable()
    try:
        alloc0 = torch.cuda.memory_allocated()
        free0, _ = torch.cuda.mem_get_info()
        for _ in range(5):
            got = pkv.paged_attention_decode_static(b.q, kc, vc, bt, sl, b.scale, out=out, lse=lse)
            assert got.data_ptr() == out.data_ptr()
        torch.cuda.synchronize()
        alloc1 = torch.cuda.memory_allocated()
        free1, _ = torch.cuda.mem_get_info()
    finally:
        gc.enable()
    assert alloc1 == alloc0
    assert free1 == free0
    assert pkv.get_device_error() == 0
    assert _close(out, ref) and _close(lse, ref_lse)
