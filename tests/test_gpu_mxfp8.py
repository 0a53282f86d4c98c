"""GPU parity for MXFP8 pools (include/pkv.h): the quantizing kv_append and
the block copy bit for bit against the oracle's pools (both planes, every
byte, 0xFF-poisoned where nothing was written); the decode element by element
against the oracle's attention over the values the oracle's own pool holds
(dequantized exactly), within |gpu - ref| <= 2e-3 + 1e-2 |ref|.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_41_gb300 import pkv
from paged_kv_cache_41_gb300 import workloads as wl

import parity_util as pu

pytestmark = pytest.mark.gpu


def _shape(b):
    return (b.num_blocks, b.block_size, b.num_kv_heads, b.head_dim)


def _pools(b):
    """Device MxPools filled through kv_append (prefill, then each sequence's
    last row), and the oracle's pools quantized from the same bf16 rows at
    slots it derives from the tables itself."""
    shape = _shape(b)
    kc = pkv.MxPool(*shape, device="cuda", fill=0xFF)
    vc = pkv.MxPool(*shape, device="cuda", fill=0xFF)
    pu.device_fill(b, kc, vc)
    hk = np.full(oracle.mxfp8_pool_bytes(*shape), 0xFF, np.uint8)
    hv = hk.copy()
    st = oracle.kv_append_mxfp8(hk, hv, shape, wl.to_numpy_storage(b.k_hist),
                                wl.to_numpy_storage(b.v_hist), pu.oracle_batch_slots(b))
    assert st == oracle.OK
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    return kc, vc, hk, hv


def _decode_and_check(b, kc, vc, hk, hv, partition_size=0, rows=None):
    dev = "cuda"
    bt = torch.from_numpy(b.block_tables).to(dev)
    sl = torch.from_numpy(b.seq_lens).to(dev)
    lse = torch.empty(b.num_seqs, b.num_q_heads, dtype=torch.float32, device=dev)
    out = pkv.paged_attention_decode(b.q, kc, vc, bt, sl, b.scale, lse=lse,
                                     partition_size=partition_size)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    shape = _shape(b)
    kf, vf = oracle.mxfp8_to_f32(hk, shape), oracle.mxfp8_to_f32(hv, shape)
    q = wl.to_numpy_storage(b.q.float())  # bf16 widened exactly
    tables, lens = b.block_tables, b.seq_lens
    if rows is not None:
        q, tables, lens = q[rows], tables[rows], lens[rows]
    ref, ref_lse = oracle.paged_decode(np.ascontiguousarray(q), kf, vf, np.ascontiguousarray(tables),
                                       np.ascontiguousarray(lens), b.scale, nthreads=pu.NTHREADS)
    got, got_lse = out.float().cpu().numpy(), lse.cpu().numpy()
    if rows is not None:
        got, got_lse = got[rows], got_lse[rows]
    pu.assert_close(got, ref, "mxfp8 out")
    pu.assert_close(got_lse, ref_lse, "mxfp8 lse")


EDGE_LENS = [0, 1, 15, 16, 31, 32, 33, 64, 100, 257, 1000]


@pytest.mark.parametrize("d,hq,hkv,p", [(128, 32, 8, 16), (64, 8, 4, 32), (128, 8, 8, 64),
                                        (128, 16, 4, 256), (64, 2, 1, 128), (128, 8, 2, 16)])
def test_append_bit_exact_and_decode(d, hq, hkv, p):
    b = wl.custom_batch(EDGE_LENS, dtype="bf16", hq=hq, hkv=hkv, d=d, p=p, seed=d + hq + p,
                        device="cuda")
    kc, vc, hk, hv = _pools(b)
    assert np.array_equal(kc.buf.cpu().numpy(), hk), "K pool bytes differ from the oracle's"
    assert np.array_equal(vc.buf.cpu().numpy(), hv), "V pool bytes differ from the oracle's"
    _decode_and_check(b, kc, vc, hk, hv)


@pytest.mark.parametrize("partition_size", [32, 128, 512])
def test_decode_split_k(partition_size):
    rng = np.random.default_rng(partition_size)
    lens = rng.integers(1, 3000, size=24)
    b = wl.custom_batch(lens, dtype="bf16", hq=32, hkv=8, d=128, p=16, seed=7, device="cuda")
    kc, vc, hk, hv = _pools(b)
    _decode_and_check(b, kc, vc, hk, hv, partition_size=partition_size)


def test_append_extreme_rows():
    # an all-zero row, tiny and huge magnitudes, one outlier per group: the
    # scale rule and the ties, bit for bit
    shape = (4, 16, 2, 128)
    kc = pkv.MxPool(*shape, device="cuda", fill=0xFF)
    vc = pkv.MxPool(*shape, device="cuda", fill=0xFF)
    g = wl.make_generator(3, "cuda")
    x = wl.randn((8, 2, 128), "bf16", g, "cuda").float()
    x[0] = 0
    x[1] *= 1e-30
    x[2] *= 1e30
    x[3, :, ::32] = 1e4
    x[4] = torch.tensor([448.0, 464.0, 465.0, 2.0 ** -9, 3 * 2.0 ** -10] * 51 + [1.0], device="cuda")[
        :256].view(2, 128)
    xb = x.to(torch.bfloat16)
    slots = torch.arange(8, dtype=torch.int64, device="cuda") * 5
    pkv.kv_append(kc, vc, xb, xb.flip(0), slots)
    hk = np.full(oracle.mxfp8_pool_bytes(*shape), 0xFF, np.uint8)
    hv = hk.copy()
    xs = wl.to_numpy_storage(xb)
    assert oracle.kv_append_mxfp8(hk, hv, shape, xs, np.ascontiguousarray(xs[::-1]),
                                  slots.cpu().numpy()) == oracle.OK
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    assert np.array_equal(kc.buf.cpu().numpy(), hk) and np.array_equal(vc.buf.cpu().numpy(), hv)


def test_block_copy_copies_both_planes():
    b = wl.custom_batch([40, 70, 5], dtype="bf16", hq=8, hkv=2, d=128, p=16, seed=11, device="cuda")
    kc, vc, hk, hv = _pools(b)
    used = set(b.block_tables[b.block_tables >= 0].tolist())
    free = [i for i in range(b.num_blocks) if i not in used]
    pairs = np.array([[b.block_tables[0, 0], free[0]], [b.block_tables[1, 4], free[1]]], np.int64)
    pkv.kv_block_copy(kc, vc, torch.from_numpy(pairs).cuda())
    shape = _shape(b)
    nb, p, hkv, d = shape
    plane = nb * p * hkv * d
    blk = p * hkv * d
    for h in (hk, hv):
        for s, t in pairs:
            h[t * blk:(t + 1) * blk] = h[s * blk:(s + 1) * blk]
            h[plane + t * blk // 32:plane + (t + 1) * blk // 32] = \
                h[plane + s * blk // 32:plane + (s + 1) * blk // 32]
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    assert np.array_equal(kc.buf.cpu().numpy(), hk) and np.array_equal(vc.buf.cpu().numpy(), hv)


def test_tree_attention_over_mxfp8_pools():
    # the tensor-core chunk-first phase takes bf16 only: every chunk goes
    # through the decode, and the merge writes bf16
    tree = [(300, 0, 6), (70, 0, 3), (45, 3, 6)] + [(r * 9 + 1, r, r + 1) for r in range(6)]
    tb = wl.prefix_tree_batch(tree, device="cuda", seed=13, hq=16, hkv=4, d=128)
    shape = (tb.num_blocks, tb.block_size, tb.num_kv_heads, tb.head_dim)
    kc = pkv.MxPool(*shape, device="cuda", fill=0xFF)
    vc = pkv.MxPool(*shape, device="cuda", fill=0xFF)
    pkv.kv_append(kc, vc, tb.k_rows, tb.v_rows, torch.from_numpy(tb.slots).cuda())
    hk = np.full(oracle.mxfp8_pool_bytes(*shape), 0xFF, np.uint8)
    hv = hk.copy()
    slots = np.concatenate([
        np.array([oracle.slot_for_position(tb.block_ids[f:], tb.block_size, t) for t in range(int(n))],
                 np.int64) for f, n, _, _ in tb.chunks])
    assert oracle.kv_append_mxfp8(hk, hv, shape, wl.to_numpy_storage(tb.k_rows),
                                  wl.to_numpy_storage(tb.v_rows), slots) == oracle.OK
    plan = pkv.chunk_tree_plan(kc, tb.chunks, tb.block_ids, tb.num_seqs, tb.num_q_heads, 0)
    lse = torch.empty(tb.num_seqs, tb.num_q_heads, dtype=torch.float32, device="cuda")
    out = pkv.chunk_tree_attention(tb.q, kc, vc, plan, tb.scale, lse=lse)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    ref, ref_lse = oracle.chunk_tree(wl.to_numpy_storage(tb.q.float()), oracle.mxfp8_to_f32(hk, shape),
                                     oracle.mxfp8_to_f32(hv, shape), tb.chunks, tb.block_ids,
                                     tb.scale)
    pu.assert_close(out.float().cpu().numpy(), ref, "tree out")
    pu.assert_close(lse.cpu().numpy(), ref_lse, "tree lse")


@pytest.mark.parametrize("p", [16, 32, 64, 128, 256])
def test_eight_heads_per_kv_head_tensor_cores(p):
    # G = 8 over MXFP8 runs only on the tensor cores (E4M3 tiles widened to bf16)
    lens = [1, 127, 128, 129, 300, 0, 1000, 33]
    b = wl.custom_batch(lens, dtype="bf16", hq=64, hkv=8, d=128, p=p, seed=17 + p, device="cuda")
    kc, vc, hk, hv = _pools(b)
    _decode_and_check(b, kc, vc, hk, hv)


@pytest.mark.parametrize("rep", range(2))
def test_tensor_core_one_stage_segments(rep):
    # every segment one 128-row stage: pieces change every stage, and the
    # widening runs one stage ahead of the MMAs
    lens = np.random.default_rng(40 + rep).integers(1, 128, size=300, endpoint=True)
    b = wl.custom_batch(lens, dtype="bf16", hq=64, hkv=8, d=128, p=16, seed=40 + rep, device="cuda")
    kc, vc, hk, hv = _pools(b)
    _decode_and_check(b, kc, vc, hk, hv)


@pytest.mark.parametrize("partition_size", [128, 512])
def test_tensor_core_split_k(partition_size):
    # pieces cut at CTA boundaries every few stages: records and the reduction
    rng = np.random.default_rng(partition_size + 1)
    lens = rng.integers(1, 3000, size=24)
    b = wl.custom_batch(lens, dtype="bf16", hq=64, hkv=8, d=128, p=16, seed=9, device="cuda")
    kc, vc, hk, hv = _pools(b)
    _decode_and_check(b, kc, vc, hk, hv, partition_size=partition_size)


def test_tree_with_eight_heads_over_mxfp8_pools():
    # sequence-first through the tensor-core MXFP8 decode: q_rows indirection
    # and states-only output
    tree = [(300, 0, 6), (70, 0, 3), (45, 3, 6)] + [(r * 9 + 1, r, r + 1) for r in range(6)]
    tb = wl.prefix_tree_batch(tree, device="cuda", seed=14, hq=64, hkv=8, d=128)
    shape = (tb.num_blocks, tb.block_size, tb.num_kv_heads, tb.head_dim)
    kc = pkv.MxPool(*shape, device="cuda", fill=0xFF)
    vc = pkv.MxPool(*shape, device="cuda", fill=0xFF)
    pkv.kv_append(kc, vc, tb.k_rows, tb.v_rows, torch.from_numpy(tb.slots).cuda())
    hk = np.full(oracle.mxfp8_pool_bytes(*shape), 0xFF, np.uint8)
    hv = hk.copy()
    slots = np.concatenate([
        np.array([oracle.slot_for_position(tb.block_ids[f:], tb.block_size, t) for t in range(int(n))],
                 np.int64) for f, n, _, _ in tb.chunks])
    assert oracle.kv_append_mxfp8(hk, hv, shape, wl.to_numpy_storage(tb.k_rows),
                                  wl.to_numpy_storage(tb.v_rows), slots) == oracle.OK
    plan = pkv.chunk_tree_plan(kc, tb.chunks, tb.block_ids, tb.num_seqs, tb.num_q_heads, 0)
    lse = torch.empty(tb.num_seqs, tb.num_q_heads, dtype=torch.float32, device="cuda")
    out = pkv.chunk_tree_attention(tb.q, kc, vc, plan, tb.scale, lse=lse)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    ref, ref_lse = oracle.chunk_tree(wl.to_numpy_storage(tb.q.float()), oracle.mxfp8_to_f32(hk, shape),
                                     oracle.mxfp8_to_f32(hv, shape), tb.chunks, tb.block_ids,
                                     tb.scale)
    pu.assert_close(out.float().cpu().numpy(), ref, "tree out")
    pu.assert_close(lse.cpu().numpy(), ref_lse, "tree lse")


@pytest.mark.parametrize("d", [128, 64])
def test_short_segments_past_the_descriptor_batches(d):
    # more than 64 stages per CTA and a piece end at nearly every stage: the
    # consumers read the next stage's descriptor (its q) at each piece end
    # while warp 0 refills the 64-entry descriptor ring with later batches;
    # every output is checked
    lens = np.random.default_rng(d + 5).integers(1, 190, size=2000, endpoint=True)
    b = wl.custom_batch(lens, dtype="bf16", hq=32, hkv=8, d=d, p=16, seed=d + 6, device="cuda")
    kc, vc, hk, hv = _pools(b)
    _decode_and_check(b, kc, vc, hk, hv)


def test_tensor_core_many_short_pieces():
    # as the bf16 test: about 150 one- or two-stage pieces per CTA through
    # the widening kernel's raw slots, bf16 buffers and descriptor ring
    lens = np.random.default_rng(78).integers(1, 190, size=2000, endpoint=True)
    b = wl.custom_batch(lens, dtype="bf16", hq=64, hkv=8, d=128, p=16, seed=78, device="cuda")
    kc, vc, hk, hv = _pools(b)
    _decode_and_check(b, kc, vc, hk, hv)


def test_tensor_core_extreme_scales():
    # scales past 2^7 (the widening's second multiply), tiny scales and
    # all-zero groups on the tensor-core path: V rows times 1e30 and 1e-30,
    # K rows times 1e5 in one sequence (its softmax turns one-hot) and 1e-30
    lens = [300, 200, 129]
    b = wl.custom_batch(lens, dtype="bf16", hq=64, hkv=8, d=128, p=16, seed=23, device="cuda")
    n = b.v_hist.shape[0]
    rows = torch.arange(n, device="cuda")
    b.v_hist[rows % 5 == 1] *= 1e30
    b.v_hist[rows % 7 == 2] *= 1e-30
    b.v_hist[rows % 11 == 3, :, 32:64] = 0
    b.k_hist[rows % 13 == 4] *= 1e-30
    k0 = rows[int(b.hist_offsets[0]):int(b.hist_offsets[1])]  # sequence 0's rows
    b.k_hist[k0[k0 % 9 == 5]] *= 1e5
    kc, vc, hk, hv = _pools(b)
    assert kc.scales.max().item() > 134 and vc.scales.max().item() > 134
    _decode_and_check(b, kc, vc, hk, hv)


@pytest.mark.parametrize("hq", [8, 16])  # 16 / 2: eight heads per kv head, the tensor cores
def test_bad_block_and_length_set_errors(hq):
    # a block id past the pool: its rows are skipped (CUDA cores) or read as
    # zero-filled boxes (tensor cores) and the error bit is set; a length past
    # the table sets its own bit
    b = wl.custom_batch([200, 20], dtype="bf16", hq=hq, hkv=2, d=128, p=16, seed=63, device="cuda")
    kc, vc, _, _ = _pools(b)
    bt = torch.from_numpy(b.block_tables).cuda()
    sl = torch.from_numpy(b.seq_lens).cuda()
    bad = bt.clone()
    bad[0, 1] = b.num_blocks + 3
    pkv.paged_attention_decode(b.q, kc, vc, bad, sl, b.scale)
    assert pkv.get_device_error() & pkv.DEVERR_BLOCK
    pkv.paged_attention_decode(b.q, kc, vc, bt, torch.tensor([200, 10_000], dtype=torch.int32,
                                                             device="cuda"), b.scale)
    assert pkv.get_device_error() & pkv.DEVERR_LENGTH
    pkv.kv_block_copy(kc, vc, torch.tensor([[0, -5]], dtype=torch.int64, device="cuda"))
    assert pkv.get_device_error() == pkv.DEVERR_BLOCK
    assert pkv.get_device_error() == 0  # read and cleared


def test_eight_heads_per_kv_head_at_head_dim_64_is_rejected():
    b = wl.custom_batch([10], dtype="bf16", hq=16, hkv=2, d=64, p=16, seed=1, device="cuda")
    kc = pkv.MxPool(*_shape(b), device="cuda")
    vc = pkv.MxPool(*_shape(b), device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_attention_decode(b.q, kc, vc, torch.from_numpy(b.block_tables).cuda(),
                                   torch.from_numpy(b.seq_lens).cuda(), b.scale)
    assert e.value.status == pkv.PKV_ERR_UNSUPPORTED


def test_llama_shaped_full_size():
    b = wl.llama_batch(device="cuda")
    shape = _shape(b)
    kc = pkv.MxPool(*shape, device="cuda", fill=0xFF)
    vc = pkv.MxPool(*shape, device="cuda", fill=0xFF)
    pu.device_fill(b, kc, vc)
    dev = "cuda"
    lse = torch.empty(b.num_seqs, b.num_q_heads, dtype=torch.float32, device=dev)
    out = pkv.paged_attention_decode(b.q, kc, vc, torch.from_numpy(b.block_tables).to(dev),
                                     torch.from_numpy(b.seq_lens).to(dev), b.scale, lse=lse)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    # the oracle quantizes every sequence into a pool of its own
    rows = np.arange(b.num_seqs)
    P = b.block_size
    tables, lens, kh, vh, slots, nxt = [], [], [], [], [], 0
    kall, vall = wl.to_numpy_storage(b.k_hist), wl.to_numpy_storage(b.v_hist)
    for r in rows:
        t = int(b.seq_lens[r])
        nblk = oracle.num_blocks(t, P)
        own = np.arange(nxt, nxt + nblk, dtype=np.int32)
        nxt += nblk
        tables.append(own)
        lens.append(t)
        lo = int(b.hist_offsets[r])
        kh.append(kall[lo:lo + t])
        vh.append(vall[lo:lo + t])
        slots.append(oracle.slots_for_positions(own[None, :], P, np.zeros(t, np.int32),
                                                np.arange(t, dtype=np.int64)))
    width = max(len(t) for t in tables)
    tb = np.full((len(rows), width), -1, np.int32)
    for i, t in enumerate(tables):
        tb[i, :len(t)] = t
    oshape = (nxt, P, b.num_kv_heads, b.head_dim)
    hk = np.zeros(oracle.mxfp8_pool_bytes(*oshape), np.uint8)
    hv = hk.copy()
    assert oracle.kv_append_mxfp8(hk, hv, oshape, np.concatenate(kh), np.concatenate(vh),
                                  np.concatenate(slots)) == oracle.OK
    q = wl.to_numpy_storage(b.q.float())[rows]
    ref, ref_lse = oracle.paged_decode(np.ascontiguousarray(q), oracle.mxfp8_to_f32(hk, oshape),
                                       oracle.mxfp8_to_f32(hv, oshape), tb,
                                       np.array(lens, np.int32), b.scale, nthreads=pu.NTHREADS)
    pu.assert_close(out.float().cpu().numpy(), ref, "llama mxfp8 out")
    pu.assert_close(lse.cpu().numpy(), ref_lse, "llama mxfp8 lse")
