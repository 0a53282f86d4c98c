"""GPU parity of attention over a prefix tree (pkv_chunk_tree_attention)
against the oracle's definition: every sequence attends to the concatenation
of the chunks covering it ("M5.3 - KV Memory Layout and Exact Reuse", 0x0BB,
0x0BE).  Outputs and LSEs element by element within |gpu - ref| <= 2e-3 +
1e-2 |ref|.  Pools start NaN-poisoned, so a ragged chunk's unused rows would
show up in the result if a kernel read them.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_41_gb300 import pkv
from paged_kv_cache_41_gb300 import workloads as wl

import parity_util as pu

pytestmark = pytest.mark.gpu


def _pools(tb, block_offset=0):
    """Device pools filled through kv_append and the oracle's own.  With
    block_offset, the device side alone relabels every block id i as
    i + block_offset in a pool that much larger (blocks below stay unused)."""
    shape = (tb.num_blocks, tb.block_size, tb.num_kv_heads, tb.head_dim)
    dt = wl.DTYPES[tb.dtype]
    kc = torch.full((block_offset + shape[0],) + shape[1:], float("nan"), dtype=dt, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    if tb.slots.size:
        dev_slots = np.where(tb.slots >= 0, tb.slots + block_offset * tb.block_size, tb.slots)
        pkv.kv_append(kc, vc, tb.k_rows, tb.v_rows, torch.from_numpy(dev_slots.astype(np.int64)).cuda())
    hk, hv = pu.host_pool(tb)
    slots = np.empty(int(tb.row_offsets[-1]), np.int64)
    for c, (first, n, _, _) in enumerate(tb.chunks):
        lo = int(tb.row_offsets[c])
        for t in range(int(n)):
            slots[lo + t] = oracle.slot_for_position(tb.block_ids[first:], tb.block_size, t)
    assert oracle.kv_append(hk, hv, wl.to_numpy_storage(tb.k_rows), wl.to_numpy_storage(tb.v_rows),
                            slots) == oracle.OK
    return kc, vc, hk, hv


def _run(tb, threshold=-1, q=None, pools=None, block_offset=0):
    kc, vc, hk, hv = pools or _pools(tb, block_offset)
    q = tb.q if q is None else q
    plan = pkv.chunk_tree_plan(kc, tb.chunks, (tb.block_ids + block_offset).astype(np.int32),
                               tb.num_seqs, tb.num_q_heads, threshold)
    lse = torch.empty(tb.num_seqs, tb.num_q_heads, dtype=torch.float32, device="cuda")
    out = pkv.chunk_tree_attention(q, kc, vc, plan, tb.scale, lse=lse)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    ref, ref_lse = oracle.chunk_tree(wl.to_numpy_storage(q), hk, hv, tb.chunks, tb.block_ids,
                                     tb.scale, nthreads=pu.NTHREADS)
    pu.assert_close(out.float().cpu().numpy(), ref, "tree out")
    pu.assert_close(lse.cpu().numpy(), ref_lse, "tree lse")
    return (kc, vc, hk, hv), plan


LOOP9 = [(2, 0, 4), (1, 0, 2), (2, 2, 4), (2, 0, 1), (1, 1, 2), (1, 2, 3), (1, 3, 4)]


@pytest.mark.parametrize("threshold", [-1, 0, 2, 4])
@pytest.mark.parametrize("scale_rows", [1, 37])
def test_loop9_shaped_tree(threshold, scale_rows):
    # the printed fixture's tree, rows scaled (ragged against 16-row blocks);
    # threshold 0 is hierarchical Hydragen, 4 runs everything sequence-first
    tree = [(n * scale_rows + (3 if scale_rows > 1 else 0), b, e) for n, b, e in LOOP9]
    tb = wl.prefix_tree_batch(tree, device="cuda", seed=11 + scale_rows, hq=8, hkv=2, d=128)
    _run(tb, threshold)


@pytest.mark.parametrize("hq,hkv,d,p", [(32, 8, 128, 16), (8, 8, 64, 16), (64, 8, 128, 16),
                                        (16, 4, 128, 64), (16, 2, 64, 128), (32, 8, 128, 256)])
def test_multi_level_tree(hq, hkv, d, p):
    tree = wl.multi_level_tree(batch=48, root_len=300, groups=3, group_len=200, leaf_lo=1,
                               leaf_hi=150, seed=hq + p)
    tb = wl.prefix_tree_batch(tree, device="cuda", seed=hq * 3 + p, hq=hq, hkv=hkv, d=d, p=p)
    _run(tb)


@pytest.mark.parametrize("threshold", [-1, 4])  # shared chunks chunk-first / all sequence-first
def test_tree_pool_past_2_31_elements(threshold):
    """Every block the tree uses lies past element 2^31 of the pool: the
    chunk-first items' block ids and the sequence-first decode's tables."""
    tree = wl.multi_level_tree(batch=40, root_len=300, groups=3, group_len=200, leaf_lo=1,
                               leaf_hi=150, seed=223)
    tb = wl.prefix_tree_batch(tree, device="cuda", seed=227, hq=32, hkv=8, d=128, p=16)
    _run(tb, threshold, block_offset=2**31 // (16 * 8 * 128) + 3)


def test_long_shared_chunk_splits_and_many_pairs():
    # a 3000-key root over 100 sequences: several key splits and query-tile
    # pairs (100 x 4 heads = 4 tiles per kv head); a 4-level path
    tree = [(3000, 0, 100), (129, 0, 50), (257, 50, 100), (64, 50, 75)]
    tree += [(1 + (r * 7) % 90, r, r + 1) for r in range(100)]
    tb = wl.prefix_tree_batch(tree, device="cuda", seed=3, hq=32, hkv=8, d=128)
    _run(tb)


def test_fp32_cache_runs_sequence_first():
    tree = [(70, 0, 5), (17, 0, 2), (9, 2, 5)] + [(r + 1, r, r + 1) for r in range(5)]
    tb = wl.prefix_tree_batch(tree, device="cuda", seed=4, hq=4, hkv=2, d=64, dtype="f32")
    _run(tb, threshold=0)


def test_uncovered_sequences_and_a_plan_reused_for_new_queries():
    # sequences 3 and 6 sit on no chunk: zero output, -inf LSE
    tree = [(90, 0, 3), (40, 4, 6), (5, 0, 1), (6, 4, 5)]
    tb = wl.prefix_tree_batch(tree, device="cuda", seed=5, hq=16, hkv=4, d=128, batch=7)
    pools, plan = _run(tb)
    q2 = wl.randn(tuple(tb.q.shape), tb.dtype, wl.make_generator(99, "cuda"), "cuda")
    lse = torch.empty(tb.num_seqs, tb.num_q_heads, dtype=torch.float32, device="cuda")
    out = pkv.chunk_tree_attention(q2, pools[0], pools[1], plan, tb.scale, lse=lse)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    ref, ref_lse = oracle.chunk_tree(wl.to_numpy_storage(q2), pools[2], pools[3], tb.chunks,
                                     tb.block_ids, tb.scale)
    pu.assert_close(out.float().cpu().numpy(), ref, "reused plan out")
    pu.assert_close(lse.cpu().numpy(), ref_lse, "reused plan lse")
    assert (out[[3, 6]] == 0).all() and torch.isinf(lse[[3, 6]]).all()


def test_tree_workload_full_size():
    # the bench's tree workload: 128 requests, a 2048-token root, 4 groups of
    # up to 1024 tokens, private leaves of 16..512
    tree = wl.multi_level_tree(batch=128, root_len=2048, groups=4, group_len=1024, leaf_lo=16,
                               leaf_hi=512, seed=6)
    tb = wl.prefix_tree_batch(tree, device="cuda", seed=6)
    _run(tb)


def test_plan_for_another_batch_is_rejected():
    tree = [(40, 0, 4), (3, 0, 1)]
    tb = wl.prefix_tree_batch(tree, device="cuda", seed=1, hq=8, hkv=2, d=64)
    kc, vc, _, _ = _pools(tb)
    plan = pkv.chunk_tree_plan(kc, tb.chunks, tb.block_ids, 5, tb.num_q_heads)
    with pytest.raises(pkv.PkvError) as e:
        pkv.chunk_tree_attention(tb.q, kc, vc, plan, tb.scale)
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG
    plan = pkv.chunk_tree_plan(kc, tb.chunks, tb.block_ids, 4, tb.num_q_heads)
    small = torch.empty(max(plan.workspace_bytes - 256, 0), dtype=torch.uint8, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.chunk_tree_attention(tb.q, kc, vc, plan, tb.scale, workspace=small)
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG
