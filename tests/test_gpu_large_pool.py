"""GPU parity on pools past 2^31 elements (bf16) or bytes (MXFP8): the
maximum-size case of the slot and block arithmetic.

"M5.3 - KV Memory Layout and Exact Reuse" (the address map, 0x0BB) widens
page ids to 64 bits before multiplying them by the row stride; the pool
here puts every block a batch uses past element (or byte) 2^31, where a
32-bit product would wrap.  The batch is relabelled on the device side only:
its block ids are shifted by OFF (and its slots by OFF * block_size) into a
pool of OFF + n blocks, while the oracle runs on the batch's own n-block pool.
A relabelling changes no result, so the device pool's last n blocks must
equal the oracle's pool bit for bit, everything below them must still hold
the poison it was filled with, and the decode must match the oracle within
|gpu - ref| <= 2e-3 + 1e-2 |ref|.  Each case holds up to 8.6 GB on the device.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_41_gb300 import pkv
from paged_kv_cache_41_gb300 import workloads as wl

import parity_util as pu

pytestmark = pytest.mark.gpu

P, HKV, D = 16, 8, 128
# first block id of the batch on the device: its first element lies past 2^31
OFF = 2**31 // (P * HKV * D) + 7
LENS = [300, 1, 17, 513, 64, 129, 0, 48]


def _shifted(b):
    tables = np.where(b.block_tables >= 0, b.block_tables + OFF, b.block_tables).astype(np.int32)
    slots = np.where(b.slots >= 0, b.slots + OFF * P, b.slots).astype(np.int64)
    return tables, slots


def _device_fill(b, kc, vc, slots):
    """The prefill rows, then each sequence's last row, at the shifted slots."""
    dev = "cuda"
    st = torch.from_numpy(slots).to(dev)
    pre = torch.from_numpy(b.prefill_rows()).to(dev)
    if pre.numel():
        pkv.kv_append(kc, vc, b.k_hist[pre], b.v_hist[pre], st[pre])
    last = torch.from_numpy(b.last_rows()[b.seq_lens > 0]).to(dev)
    if last.numel():
        pkv.kv_append(kc, vc, b.k_hist[last], b.v_hist[last], st[last])


def _decode(b, kc, vc, tables):
    dev = "cuda"
    lse = torch.empty(b.num_seqs, b.num_q_heads, dtype=torch.float32, device=dev)
    out = pkv.paged_attention_decode(b.q, kc, vc, torch.from_numpy(tables).to(dev),
                                     torch.from_numpy(b.seq_lens).to(dev), b.scale, lse=lse)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _bf16_bits(t):
    return t.contiguous().view(torch.int16)


@pytest.mark.parametrize("hq", [32, 64])  # 64 / 8: the tensor-core decode
def test_bf16_pool_past_2_31_elements(hq):
    b = wl.custom_batch(LENS, dtype="bf16", hq=hq, hkv=HKV, d=D, p=P, seed=131 + hq, device="cuda")
    n = b.num_blocks
    assert OFF * P * HKV * D > 2**31
    tables, slots = _shifted(b)
    kc = torch.full((OFF + n, P, HKV, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    _device_fill(b, kc, vc, slots)
    hk, hv = pu.host_pool(b)
    pu.oracle_fill(b, hk, hv)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    assert pu.pools_equal_bytes(kc[OFF:], hk) and pu.pools_equal_bytes(vc[OFF:], hv)
    poison = torch.full((), float("nan"), dtype=torch.bfloat16, device="cuda").view(torch.int16)
    assert bool((_bf16_bits(kc[:OFF]) == poison).all()) and bool((_bf16_bits(vc[:OFF]) == poison).all())

    out, lse = _decode(b, kc, vc, tables)
    ref, ref_lse = pu.oracle_decode(b, hk, hv)
    pu.assert_close(out, ref, "out")
    pu.assert_close(lse, ref_lse, "lse")

    # block copies high -> high (oracle ids: minus OFF) and high -> block 3
    used = sorted(set(b.block_tables[b.block_tables >= 0].tolist()))
    free = [i for i in range(n) if i not in set(used)]
    pairs = np.array([(used[0], free[0]), (used[-1], free[1])], np.int64)
    dev_pairs = np.concatenate([pairs + OFF, [[used[1] + OFF, 3]]]).astype(np.int64)
    pkv.kv_block_copy(kc, vc, torch.from_numpy(dev_pairs).cuda())
    assert oracle.kv_block_copy(hk, hv, pairs) == oracle.OK
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    assert pu.pools_equal_bytes(kc[OFF:], hk) and pu.pools_equal_bytes(vc[OFF:], hv)
    assert pu.pools_equal_bytes(kc[3:4], hk[used[1]:used[1] + 1])
    assert pu.pools_equal_bytes(vc[3:4], hv[used[1]:used[1] + 1])
    assert bool((_bf16_bits(kc[:3]) == poison).all()) and bool((_bf16_bits(kc[4:OFF]) == poison).all())


@pytest.mark.parametrize("hq", [32, 64])  # 64 / 8: the tensor-core MXFP8 decode
def test_mxfp8_pool_past_2_31_bytes(hq):
    b = wl.custom_batch(LENS, dtype="bf16", hq=hq, hkv=HKV, d=D, p=P, seed=137 + hq, device="cuda")
    n = b.num_blocks
    assert OFF * P * HKV * D > 2**31  # one byte per element
    tables, slots = _shifted(b)
    kc = pkv.MxPool(OFF + n, P, HKV, D, device="cuda", fill=0xFF)
    vc = pkv.MxPool(OFF + n, P, HKV, D, device="cuda", fill=0xFF)
    _device_fill(b, kc, vc, slots)
    shape = (n, P, HKV, D)
    hk = np.full(oracle.mxfp8_pool_bytes(*shape), 0xFF, np.uint8)
    hv = hk.copy()
    assert oracle.kv_append_mxfp8(hk, hv, shape, wl.to_numpy_storage(b.k_hist),
                                  wl.to_numpy_storage(b.v_hist), pu.oracle_batch_slots(b)) == oracle.OK
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    plane = n * P * HKV * D
    for dev_pool, host in ((kc, hk), (vc, hv)):
        assert np.array_equal(dev_pool.elements[OFF:].cpu().numpy().reshape(-1), host[:plane])
        assert np.array_equal(dev_pool.scales[OFF:].cpu().numpy().reshape(-1), host[plane:])
        assert bool((dev_pool.elements[:OFF] == 0xFF).all()) and bool((dev_pool.scales[:OFF] == 0xFF).all())

    out, lse = _decode(b, kc, vc, tables)
    kf, vf = oracle.mxfp8_to_f32(hk, shape), oracle.mxfp8_to_f32(hv, shape)
    q = wl.to_numpy_storage(b.q.float())
    ref, ref_lse = oracle.paged_decode(np.ascontiguousarray(q), kf, vf, b.block_tables, b.seq_lens,
                                       b.scale, nthreads=pu.NTHREADS)
    pu.assert_close(out, ref, "out")
    pu.assert_close(lse, ref_lse, "lse")
