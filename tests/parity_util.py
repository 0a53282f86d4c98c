"""Helpers shared by the GPU parity tests: run a workload through the device
path (libpkv via its binding) and through the CPU oracle on the same inputs.

The oracle side never sees a value produced by the device path: it fills its
own pool from the generator's logical rows, at slots it derives itself from
the block tables.
"""
import os

import numpy as np
import torch

import oracle
from paged_kv_cache_41_gb300 import pkv
from paged_kv_cache_41_gb300 import workloads as wl

# attention tolerance of the problem statement: |gpu - ref| <= 2e-3 + 1e-2 |ref|
ATOL, RTOL = 2e-3, 1e-2

NTHREADS = max(1, len(os.sched_getaffinity(0)))


def assert_close(gpu, ref, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    both_inf = np.isinf(ref) & (gpu == ref)
    with np.errstate(invalid="ignore"):
        err = np.where(both_inf, 0.0, np.abs(gpu - ref))
    bound = ATOL + RTOL * np.where(both_inf, 0.0, np.abs(ref))
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance; first at {tuple(i)}: "
                             f"gpu={gpu[tuple(i)]!r} ref={ref[tuple(i)]!r}")


def oracle_batch_slots(b: wl.PagedBatch) -> np.ndarray:
    """The oracle's slot for every history row, in history order."""
    lens = b.seq_lens.astype(np.int64)
    rows = np.repeat(np.arange(b.num_seqs, dtype=np.int32), lens)
    pos = np.arange(int(lens.sum()), dtype=np.int64) - np.repeat(b.hist_offsets[:-1], lens)
    return oracle.slots_for_positions(b.block_tables, b.block_size, rows, pos)


def device_pool(b, device="cuda"):
    shape = (b.num_blocks, b.block_size, b.num_kv_heads, b.head_dim)
    dt = wl.DTYPES[b.dtype]
    kc = torch.full(shape, float("nan"), dtype=dt, device=device)
    vc = torch.full(shape, float("nan"), dtype=dt, device=device)
    return kc, vc


def host_pool(b):
    shape = (b.num_blocks, b.block_size, b.num_kv_heads, b.head_dim)
    if b.dtype == "f32":
        return np.full(shape, np.nan, np.float32), np.full(shape, np.nan, np.float32)
    return np.full(shape, 0x7FC0, np.uint16), np.full(shape, 0x7FC0, np.uint16)


def device_fill(b: wl.PagedBatch, kc, vc):
    """Prefill every history row but the last through kv_append, then the step's
    last rows through a second kv_append (the decode step's append)."""
    dev = kc.device
    slots = torch.from_numpy(b.slots).to(dev)
    pre = torch.from_numpy(b.prefill_rows()).to(dev)
    if pre.numel():
        pkv.kv_append(kc, vc, b.k_hist[pre], b.v_hist[pre], slots[pre])
    last = b.last_rows()[b.seq_lens > 0]
    lt = torch.from_numpy(last).to(dev)
    if lt.numel():
        pkv.kv_append(kc, vc, b.k_hist[lt], b.v_hist[lt], slots[lt])


def oracle_fill(b: wl.PagedBatch, kc, vc):
    kh, vh = wl.to_numpy_storage(b.k_hist), wl.to_numpy_storage(b.v_hist)
    st = oracle.kv_append(kc, vc, kh, vh, oracle_batch_slots(b))
    assert st == oracle.OK


def device_decode(b: wl.PagedBatch, kc, vc, partition_size=0):
    dev = kc.device
    bt = torch.from_numpy(b.block_tables).to(dev)
    sl = torch.from_numpy(b.seq_lens).to(dev)
    lse = torch.empty(b.num_seqs, b.num_q_heads, dtype=torch.float32, device=dev)
    out = pkv.paged_attention_decode(b.q, kc, vc, bt, sl, b.scale, lse=lse,
                                     partition_size=partition_size)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def oracle_decode(b: wl.PagedBatch, kc, vc, rows=None):
    q = wl.to_numpy_storage(b.q)
    bt, sl = b.block_tables, b.seq_lens
    if rows is not None:
        q, bt, sl = q[rows], bt[rows], sl[rows]
    return oracle.paged_decode(np.ascontiguousarray(q), kc, vc, np.ascontiguousarray(bt),
                               np.ascontiguousarray(sl), b.scale, nthreads=NTHREADS)


def pools_equal_bytes(dev_tensor, host_array) -> bool:
    d = dev_tensor.contiguous().cpu()
    if d.dtype == torch.bfloat16:
        d = d.view(torch.int16).numpy().view(np.uint16)
    else:
        d = d.view(torch.int32).numpy().view(np.float32)
    return np.array_equal(d.view(np.uint8), host_array.view(np.uint8))
