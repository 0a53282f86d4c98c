"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks the oracle against something the pages print (fixtures in
tests/golden/, each with its citation), a closed form, an invariant the pages
state, a special case that reduces to a library routine, or brute force on
tiny inputs.  No expected value here comes from the CUDA path.
"""
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
from oracle import prefix_tree
from paged_kv_cache_41_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


# ------------------------------------------------------------------ index math
def test_block_counts_printed_in_pages():
    rows = _rows("block_counts.txt")
    assert len(rows) == 5
    for t, p, nb, tail in rows:
        assert oracle.num_blocks(int(t), int(p)) == int(nb)
        if tail != "-":
            assert oracle.tail_rows(int(t), int(p)) == int(tail)


def test_block_count_edges():
    # T = k*P fills its last block; T = k*P + 1 spills one row; T = 0 has none
    assert oracle.num_blocks(32, 16) == 2 and oracle.tail_rows(32, 16) == 16
    assert oracle.num_blocks(33, 16) == 3 and oracle.tail_rows(33, 16) == 1
    assert oracle.num_blocks(0, 16) == 0 and oracle.tail_rows(0, 16) == 0
    assert oracle.num_blocks(1, 16) == 1 and oracle.tail_rows(1, 16) == 1


def test_checked_address_trace():
    kv = {r[0]: r[1:] for r in _rows("address_trace.txt") if r[0] != "slot_id"}
    shape = [int(x) for x in kv["shape"]]
    coord = [int(x) for x in kv["coord"]]
    # the printed strides are the offsets of the unit coordinates
    for a, stride in enumerate(int(x) for x in kv["strides"]):
        unit = [0] * len(shape)
        unit[a] = 1
        assert oracle.row_major_offset(shape, unit) == stride
    e = oracle.row_major_offset(shape, coord)
    assert e == int(kv["element_offset"][0])
    assert int(kv["scalar_bytes"][0]) * e == int(kv["byte_offset"][0])
    assert int(kv["k_base"][0]) + int(kv["byte_offset"][0]) == int(kv["byte_address"][0])
    # the slot id and the byte address are different quantities
    assert oracle.slot_id(6, 16, 0) != int(kv["byte_address"][0])
    # an out-of-range coordinate is rejected
    assert oracle.row_major_offset(shape, [0, 8, 0, 1, 5]) == -1


def test_slot_ids_printed_in_pages():
    for r in _rows("address_trace.txt"):
        if r[0] == "slot_id":
            slot, p, off, want = map(int, r[1:])
            assert oracle.slot_id(slot, p, off) == want


def test_resolve_visibility_printed_in_pages():
    nb = 64
    table = [11, 40, 7]
    for ctx, p, tok, expect, lb, off in _rows("visibility.txt"):
        st, blk, o = oracle.resolve(table, int(ctx), int(p), nb, int(tok))
        if expect == "ok":
            assert st == oracle.OK
            assert blk == table[int(lb)] and o == int(off)
        else:
            assert st == oracle.REJECT_VISIBILITY


def test_resolve_rejection_order():
    # visibility is checked before the table bound, the table bound before identity
    assert oracle.resolve([3], 16, 16, 8, 20)[0] == oracle.REJECT_VISIBILITY
    assert oracle.resolve([3], 40, 16, 8, 20)[0] == oracle.REJECT_TABLE
    assert oracle.resolve([3, 99], 40, 16, 8, 20)[0] == oracle.REJECT_PHYSICAL
    assert oracle.resolve([3, -1], 40, 16, 8, 20)[0] == oracle.REJECT_PHYSICAL
    assert oracle.resolve([3, 5], 40, 16, 8, 20)[:2] == (oracle.OK, 5)


@pytest.mark.parametrize("table", [[3, 8, 1], [7, 2, 19]])
def test_slot_mapping_of_the_35_token_example(table):
    # "7. Memory Management and Local Model State", section "Logical tokens,
    # physical blocks", draws the 35-token sequence twice with different
    # placements: its flowchart maps logical blocks 0, 1, 2 to physical blocks
    # 3, 8, 1, and the position ruler below it to 7, 2, 19.  Either table must
    # give the same slots: whole physical row ranges for the two full blocks
    # and the first three rows of the third.
    a, b, c = table
    expect = (list(range(a * 16, (a + 1) * 16)) + list(range(b * 16, (b + 1) * 16))
              + list(range(c * 16, c * 16 + 3)))
    got = [oracle.slot_for_position(table, 16, t) for t in range(35)]
    assert got == expect


def test_batched_slots_equal_enumerated_row_ranges():
    # the batched form against the slots enumerated as whole physical row
    # ranges of each request's blocks, for a ragged, shuffled batch
    rng = np.random.default_rng(7)
    p = 16
    ids = rng.permutation(200).astype(np.int32)
    lens = [35, 1, 16, 100, 0, 47]
    tables = np.full((len(lens), 8), -1, np.int32)
    expect, rows, pos, nxt = [], [], [], 0
    for r, t in enumerate(lens):
        n = -(-t // p)
        tables[r, :n] = ids[nxt:nxt + n]
        nxt += n
        slots = np.concatenate([np.arange(b * p, (b + 1) * p) for b in tables[r, :n]] or [[]])
        expect.extend(slots[:t].tolist())
        rows += [r] * t
        pos += list(range(t))
    order = rng.permutation(len(pos))
    got = oracle.slots_for_positions(tables, p, np.array(rows)[order], np.array(pos)[order])
    assert got.tolist() == np.array(expect, np.int64)[order].tolist()
    with pytest.raises(ValueError):
        oracle.slots_for_positions(tables, p, [0], [8 * p])  # past the table


def test_slot_ids_widen_to_int64():
    # a page id whose slot exceeds int32 range ("widen page ids to int64 before
    # multiplying by pool strides")
    big = 2**31 - 5
    assert oracle.slot_for_position([big], 64, 63) == big * 64 + 63


# ------------------------------------------------------------------ append / copy
def _rand_cache(nb, p, hkv, d, dtype, rng):
    if dtype == "f32":
        return rng.standard_normal((nb, p, hkv, d)).astype(np.float32)
    return rng.integers(0, 2**16, size=(nb, p, hkv, d), dtype=np.uint16)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_append_matches_fancy_index_scatter(dtype):
    rng = np.random.default_rng(7)
    nb, p, hkv, d = 6, 16, 2, 8
    kc, vc = _rand_cache(nb, p, hkv, d, dtype, rng), _rand_cache(nb, p, hkv, d, dtype, rng)
    n = 20
    slots = rng.choice(nb * p, size=n, replace=False).astype(np.int64)
    slots[[3, 11]] = -1  # skip sentinel
    k = _rand_cache(n, hkv, d, 1, dtype, rng).reshape(n, hkv, d)
    v = _rand_cache(n, hkv, d, 1, dtype, rng).reshape(n, hkv, d)
    ek, ev = kc.copy().reshape(nb * p, hkv, d), vc.copy().reshape(nb * p, hkv, d)
    keep = slots >= 0
    ek[slots[keep]] = k[keep]
    ev[slots[keep]] = v[keep]
    assert oracle.kv_append(kc, vc, k, v, slots) == oracle.OK
    assert np.array_equal(kc.reshape(nb * p, hkv, d).view(np.uint8), ek.view(np.uint8))
    assert np.array_equal(vc.reshape(nb * p, hkv, d).view(np.uint8), ev.view(np.uint8))


def test_append_rejects_slot_past_pool():
    rng = np.random.default_rng(8)
    kc = np.zeros((2, 16, 1, 4), np.float32)
    vc = np.zeros_like(kc)
    k = rng.standard_normal((2, 1, 4)).astype(np.float32)
    st = oracle.kv_append(kc, vc, k, k, np.array([5, 32], np.int64))
    assert st == oracle.BAD_SLOT
    assert np.array_equal(kc[0, 5], k[0]) and not kc[1].any()


def test_block_copy_matches_slicing_in_order():
    rng = np.random.default_rng(9)
    nb, p, hkv, d = 8, 16, 2, 4
    kc = _rand_cache(nb, p, hkv, d, "bf16", rng)
    vc = _rand_cache(nb, p, hkv, d, "bf16", rng)
    ek, ev = kc.copy(), vc.copy()
    pairs = [(1, 4), (4, 6), (2, 0)]
    for s, t in pairs:
        ek[t] = ek[s]
        ev[t] = ev[s]
    assert oracle.kv_block_copy(kc, vc, pairs) == oracle.OK
    assert np.array_equal(kc, ek) and np.array_equal(vc, ev)
    assert np.array_equal(kc[6], kc[1])  # chained copies apply in order
    assert oracle.kv_block_copy(kc, vc, [(0, 8)]) == oracle.BAD_BLOCK


# ------------------------------------------------------------------ decode
def _oracle_pool_from_batch(b: wl.PagedBatch):
    """Fill an oracle-side pool from the logical history, with slots derived by
    the oracle's own translation of the block tables."""
    kh, vh = wl.to_numpy_storage(b.k_hist), wl.to_numpy_storage(b.v_hist)
    fill = np.nan if b.dtype == "f32" else 0x7FC0  # NaN poison in unused rows
    shape = (b.num_blocks, b.block_size, b.num_kv_heads, b.head_dim)
    kc = np.full(shape, fill, dtype=kh.dtype)
    vc = np.full(shape, fill, dtype=kh.dtype)
    slots = np.concatenate([
        np.array([oracle.slot_for_position(b.block_tables[r], b.block_size, t)
                  for t in range(int(b.seq_lens[r]))], dtype=np.int64)
        for r in range(b.num_seqs)]) if b.num_seqs else np.zeros(0, np.int64)
    assert oracle.kv_append(kc, vc, kh, vh, slots) == oracle.OK
    return kc, vc


def _scipy_attention(b: wl.PagedBatch):
    """Attention over the logical (never paged) history with library routines."""
    kh, vh, q = b.k_hist.double().numpy(), b.v_hist.double().numpy(), b.q.double().numpy()
    g = b.num_q_heads // b.num_kv_heads
    out = np.zeros((b.num_seqs, b.num_q_heads, b.head_dim))
    lse = np.full((b.num_seqs, b.num_q_heads), -np.inf)
    for r in range(b.num_seqs):
        lo, hi = b.hist_offsets[r], b.hist_offsets[r + 1]
        if hi == lo:
            continue
        for h in range(b.num_q_heads):
            s = b.scale * (kh[lo:hi, h // g, :] @ q[r, h])
            lse[r, h] = logsumexp(s)
            out[r, h] = np.exp(s - lse[r, h]) @ vh[lo:hi, h // g, :]
    return out, lse


@pytest.mark.parametrize("maker", ["tiny", "bf16_small"])
def test_decode_matches_library_softmax_on_logical_history(maker):
    if maker == "tiny":
        b = wl.tiny_batch()
    else:
        b = wl.custom_batch([1, 15, 16, 17, 40, 0, 64], dtype="bf16", hq=8, hkv=2, d=32, p=16,
                            seed=11)
    kc, vc = _oracle_pool_from_batch(b)
    out, lse = oracle.paged_decode(wl.to_numpy_storage(b.q), kc, vc, b.block_tables,
                                   b.seq_lens, b.scale)
    ref, ref_lse = _scipy_attention(b)
    assert np.isfinite(out).all()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_decode_permutation_invariance_is_bitwise():
    b = wl.custom_batch([37, 5, 80], dtype="bf16", hq=4, hkv=2, d=16, p=16, seed=12)
    kc, vc = _oracle_pool_from_batch(b)
    q = wl.to_numpy_storage(b.q)
    out, lse = oracle.paged_decode(q, kc, vc, b.block_tables, b.seq_lens, b.scale)
    perm = np.random.default_rng(3).permutation(b.num_blocks)  # new id of old block i
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    bt2 = np.where(b.block_tables >= 0, perm[np.maximum(b.block_tables, 0)], -1).astype(np.int32)
    out2, lse2 = oracle.paged_decode(q, kc2, vc2, bt2, b.seq_lens, b.scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_table_expansion_printed_in_pages():
    rows = _rows("table_expansion.txt")
    assert len(rows) == 2
    for pa, pk, ids, kernel in rows:
        q = int(pa) // int(pk)
        if ids == "*":
            assert oracle.expand_table(np.array([[9]], np.int32), q).shape == (1, int(kernel))
        else:
            got = oracle.expand_table(np.array([int(x) for x in ids.split(",")], np.int32), q)
            assert got.tolist() == [int(x) for x in kernel.split(",")]


def test_table_expansion_padding_identity_and_order():
    t = np.array([[5, 0, -1], [2, -1, -1]], np.int32)
    assert np.array_equal(oracle.expand_table(t, 1), t)
    e = oracle.expand_table(t, 3)
    assert e.tolist() == [[15, 16, 17, 0, 1, 2, -1, -1, -1], [6, 7, 8, -1, -1, -1, -1, -1, -1]]
    with pytest.raises(ValueError):
        oracle.expand_table(t, 0)
    with pytest.raises(ValueError):  # 2^30 * 2 does not fit an int32 id
        oracle.expand_table(np.array([1 << 30], np.int32), 2)


@pytest.mark.parametrize("pa,pk", [(32, 16), (64, 16), (256, 64), (16, 16)])
def test_decode_through_expanded_table_is_bitwise_equal(pa, pk):
    """[M5.3] 0x0AC: the payload is not duplicated -- the same pool bytes,
    viewed as q-fold more blocks of P_k rows and read through the expanded
    table, give the very same attention (bitwise, in the oracle)."""
    b = wl.custom_batch([37, 1, 200, 64, 0], dtype="bf16", hq=4, hkv=2, d=16, p=pa, seed=13)
    kc, vc = _oracle_pool_from_batch(b)
    q = wl.to_numpy_storage(b.q)
    out, lse = oracle.paged_decode(q, kc, vc, b.block_tables, b.seq_lens, b.scale)
    r = pa // pk
    view = (b.num_blocks * r, pk, b.num_kv_heads, b.head_dim)
    out2, lse2 = oracle.paged_decode(q, kc.reshape(view), vc.reshape(view),
                                     oracle.expand_table(b.block_tables, r), b.seq_lens, b.scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def _one_seq(k, v, q, scale, p=4):
    """Pack one sequence (rows [T, 1, D]) into a pool with reversed block order."""
    t, d = k.shape[0], k.shape[-1]
    n = max(1, oracle.num_blocks(t, p))
    kc = np.full((n, p, 1, d), np.nan, np.float32)
    vc = np.full((n, p, 1, d), np.nan, np.float32)
    table = np.arange(n - 1, -1, -1, dtype=np.int32)
    slots = np.array([oracle.slot_for_position(table, p, i) for i in range(t)], np.int64)
    oracle.kv_append(kc, vc, k.reshape(t, 1, d), v.reshape(t, 1, d), slots)
    return oracle.paged_decode(q.reshape(1, 1, d), kc, vc, table.reshape(1, -1),
                               np.array([t], np.int32), scale)


def test_single_token_returns_its_value_row():
    rng = np.random.default_rng(1)
    k, v, q = (rng.standard_normal((1, 8)).astype(np.float32) for _ in range(3))
    out, lse = _one_seq(k, v, q, 0.3)
    assert np.array_equal(out[0, 0], v[0].astype(np.float64))
    assert lse[0, 0] == pytest.approx(0.3 * float(np.dot(q[0].astype(np.float64), k[0])), rel=1e-15)


def test_equal_keys_average_the_values():
    rng = np.random.default_rng(2)
    t = 11
    k = np.repeat(rng.standard_normal((1, 8)).astype(np.float32), t, axis=0)
    v = rng.standard_normal((t, 8)).astype(np.float32)
    q = rng.standard_normal((1, 8)).astype(np.float32)
    out, lse = _one_seq(k, v, q, 0.5)
    np.testing.assert_allclose(out[0, 0], v.astype(np.float64).mean(axis=0), rtol=0, atol=1e-15)
    s = 0.5 * float(np.dot(q[0].astype(np.float64), k[0]))
    assert lse[0, 0] == pytest.approx(s + math.log(t), rel=1e-14)


def test_two_token_closed_form():
    # softmax of two scores is the logistic function of their difference
    rng = np.random.default_rng(4)
    k, v = rng.standard_normal((2, 6)).astype(np.float32), rng.standard_normal((2, 6)).astype(np.float32)
    q = rng.standard_normal((1, 6)).astype(np.float32)
    scale = 0.7
    s0, s1 = (scale * float(np.dot(q[0].astype(np.float64), k[i])) for i in range(2))
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))
    want = v[0].astype(np.float64) * (1 - w1) + v[1].astype(np.float64) * w1
    out, lse = _one_seq(k, v, q, scale)
    np.testing.assert_allclose(out[0, 0], want, rtol=0, atol=1e-14)
    assert lse[0, 0] == pytest.approx(max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))), rel=1e-14)


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(5)
    t, d = 9, 4
    k = np.zeros((t, d), np.float32)
    k[6] = 1.0
    v = rng.standard_normal((t, d)).astype(np.float32)
    q = np.ones((1, d), np.float32)
    out, _ = _one_seq(k, v, q, 200.0)  # scores 800 vs 0: the other weights are e^-800
    assert np.array_equal(out[0, 0], v[6].astype(np.float64))


def test_gqa_groups_are_contiguous():
    # q heads h use kv head h // (Hq / Hkv): with Hq=4, Hkv=2 heads 0,1 read kv
    # head 0 (all values +1) and heads 2,3 read kv head 1 (all values -1)
    t, d, p = 5, 4, 4
    rng = np.random.default_rng(6)
    k = rng.standard_normal((t, 2, d)).astype(np.float32)
    v = np.empty((t, 2, d), np.float32)
    v[:, 0], v[:, 1] = 1.0, -1.0
    kc = np.zeros((2, p, 2, d), np.float32)
    vc = np.zeros_like(kc)
    table = np.array([[1, 0]], np.int32)
    oracle.kv_append(kc, vc, k, v, np.array([oracle.slot_for_position(table[0], p, i)
                                             for i in range(t)], np.int64))
    q = rng.standard_normal((1, 4, d)).astype(np.float32)
    out, _ = oracle.paged_decode(q, kc, vc, table, np.array([t], np.int32), 0.5)
    np.testing.assert_allclose(out[0, :2], 1.0, atol=1e-15)
    np.testing.assert_allclose(out[0, 2:], -1.0, atol=1e-15)


def test_empty_sequence_is_zero_with_minus_inf_lse():
    kc = np.zeros((2, 16, 1, 4), np.float32)
    out, lse = oracle.paged_decode(np.ones((1, 1, 4), np.float32), kc, kc,
                                   np.full((1, 1), -1, np.int32), np.array([0], np.int32), 1.0)
    assert not out.any() and lse[0, 0] == -np.inf


def test_stale_tail_rows_are_never_read():
    # NaN-poisoned unused rows (tail of the last block, unused blocks) must not
    # reach the result; the clean pool gives the same bits.
    b = wl.custom_batch([35, 100, 16, 1], dtype="f32", hq=4, hkv=2, d=64, p=16, num_blocks=32,
                        seed=1, scale=0.125)
    kc, vc = _oracle_pool_from_batch(b)  # NaN-filled outside the history
    q = wl.to_numpy_storage(b.q)
    out, lse = oracle.paged_decode(q, kc, vc, b.block_tables, b.seq_lens, b.scale)
    assert np.isfinite(out).all()
    kc0, vc0 = np.nan_to_num(kc, nan=0.0), np.nan_to_num(vc, nan=0.0)
    out0, lse0 = oracle.paged_decode(q, kc0, vc0, b.block_tables, b.seq_lens, b.scale)
    assert np.array_equal(out, out0) and np.array_equal(lse, lse0)


# ------------------------------------------------------------------ shared prefix
def _shared_prefix_pools(sp: wl.SharedPrefixBatch):
    pk, pv = wl.to_numpy_storage(sp.parent_k), wl.to_numpy_storage(sp.parent_v)
    ck, cv = wl.to_numpy_storage(sp.child_k), wl.to_numpy_storage(sp.child_v)
    shape = (sp.num_blocks, sp.block_size, sp.num_kv_heads, sp.head_dim)
    kc = np.full(shape, 0x7FC0, np.uint16)
    vc = np.full(shape, 0x7FC0, np.uint16)
    n_par = sp.prefix_len + sp.shared_tail
    ps = np.array([oracle.slot_for_position(sp.parent_table, sp.block_size, t)
                   for t in range(n_par)], np.int64)
    oracle.kv_append(kc, vc, pk, pv, ps)
    assert oracle.kv_block_copy(kc, vc, sp.cow_pairs) == oracle.OK
    npre = sp.prefix_len // sp.block_size
    for r in range(sp.num_seqs):
        table = np.concatenate([sp.prefix_block_ids, sp.suffix_tables[r]])
        lo, hi = sp.child_offsets[r], sp.child_offsets[r + 1]
        cs = np.array([oracle.slot_for_position(table, sp.block_size, n_par + i)
                       for i in range(hi - lo)], np.int64)
        oracle.kv_append(kc, vc, np.ascontiguousarray(ck[lo:hi]), np.ascontiguousarray(cv[lo:hi]), cs)
    return kc, vc, npre


def test_shared_prefix_equals_private_copies():
    sp = wl.shared_prefix_batch(batch=6, prefix_len=64, shared_tail=5, suffix_lo=5, suffix_hi=40,
                                hq=4, hkv=2, d=16, p=16, seed=21)
    kc, vc, npre = _shared_prefix_pools(sp)
    q = wl.to_numpy_storage(sp.q)
    out, lse = oracle.shared_prefix(q, kc, vc, sp.prefix_block_ids, sp.prefix_len,
                                    sp.suffix_tables, sp.suffix_lens, sp.scale)
    # private layout: every request owns a copy of the prefix blocks
    nb = sp.num_blocks
    extra = sp.num_seqs * npre
    kc2 = np.concatenate([kc, np.zeros((extra,) + kc.shape[1:], kc.dtype)])
    vc2 = np.concatenate([vc, np.zeros((extra,) + vc.shape[1:], vc.dtype)])
    tables, lens = [], []
    for r in range(sp.num_seqs):
        own = np.arange(nb + r * npre, nb + (r + 1) * npre, dtype=np.int32)
        kc2[own], vc2[own] = kc[sp.prefix_block_ids], vc[sp.prefix_block_ids]
        tables.append(np.concatenate([own, sp.suffix_tables[r]]))
        lens.append(sp.prefix_len + sp.suffix_lens[r])
    out2, lse2 = oracle.paged_decode(q, kc2, vc2, np.array(tables, np.int32),
                                     np.array(lens, np.int32), sp.scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)
    # and the CoW left every child with private copies of the shared tail rows
    assert len(sp.cow_pairs) == sp.num_seqs - 1


def _lse_merge(parts):
    """Hydragen-coordinate merge of (O_p, LSE_p) partitions, numpy fp64."""
    lses = np.array([l for _, l in parts])
    mx = lses.max()
    w = np.exp(lses - mx)
    o = sum(wi * oi for wi, (oi, _) in zip(w, parts)) / w.sum()
    return o, mx + np.log(w.sum())


def _loop9():
    """The printed fixture: chunk (name, rows, begin, end) in tree order, the
    shapes and the ledger."""
    rows = _rows("chunk_tree_loop9.txt")
    chunks = [(r[1], int(r[2]), int(r[3]), int(r[4])) for r in rows if r[0] == "chunk"]
    shape = {r[1]: int(r[2]) for r in rows if r[0] == "shape"}
    ledger = {r[1]: int(r[2]) for r in rows if r[0] == "ledger"}
    bound = float(next(r[2] for r in rows if r[0] == "bound"))
    return chunks, shape, ledger, bound


def _loop9_dense(seed):
    chunks, shape, _, _ = _loop9()
    rng = np.random.default_rng(seed)
    dense = [prefix_tree.Chunk(rng.standard_normal((n, shape["d_qk"])),
                               rng.standard_normal((n, shape["d_v"])), b, e)
             for _, n, b, e in chunks]
    return rng.standard_normal((shape["B"], shape["d_qk"])), dense, shape


def test_loop9_ledger_printed_in_pages():
    chunks, shape, want, _ = _loop9()
    _, dense, _ = _loop9_dense(0)
    got = prefix_tree.ledger(dense, shape["d_qk"], shape["d_v"], elem_bytes=2, state_bytes=4,
                             threshold=1)
    assert got == want
    # the paths the intervals imply: S0 C0,C1,C3; S1 C0,C1,C4; S2 C0,C2,C5; S3 C0,C2,C6
    names = [c[0][:2] for c in chunks]
    assert [[names[i] for i in prefix_tree.path(dense, r)] for r in range(4)] == [
        ["C0", "C1", "C3"], ["C0", "C1", "C4"], ["C0", "C2", "C5"], ["C0", "C2", "C6"]]


def test_loop9_row_ledger_through_a_paged_pool():
    # the same counts from the oracle's slot ledger: page the tree with block
    # size 1 (one pool block per chunk row) and count logical vs unique slots
    chunks, _, want, _ = _loop9()
    ids, nxt = [], 0
    for _, n, _, _ in chunks:
        ids.append(list(range(nxt, nxt + n)))
        nxt += n
    tables, lens = [], []
    for r in range(4):
        row = sum((ids[i] for i, c in enumerate(chunks) if c[2] <= r < c[3]), [])
        tables.append(row + [-1] * (8 - len(row)))
        lens.append(len(row))
    lo, un = oracle.row_ledger(np.array(tables, np.int32), np.array(lens, np.int32), nxt, 1)
    assert (lo, un, lo - un) == (want["logical_pairs"], want["physical_rows"], want["saved_reads"])


@pytest.mark.parametrize("seed", range(40))
def test_loop9_three_schedules_agree(seed):
    # 0x0BE: both partitioned schedules match the monolithic row to rounding
    # (2.3e-16 absolute on the page's values).  These are other seeded values
    # with |o| up to ~3, so the bound is scaled by (1 + |ref|) and given a
    # factor of 4.
    _, _, _, bound = _loop9()
    Q, dense, shape = _loop9_dense(seed)
    scale = 1.0 / math.sqrt(shape["d_qk"])
    o0, l0 = prefix_tree.monolithic(Q, dense, scale)
    o1, l1 = prefix_tree.hydragen(Q, dense, scale)
    o2, l2, n_partial = prefix_tree.chunk_attention(Q, dense, scale, threshold=1)
    assert n_partial == 8
    tol = 4 * bound
    for o, l in ((o1, l1), (o2, l2)):
        assert np.all(np.abs(o - o0) <= tol * (1 + np.abs(o0)))
        assert np.all(np.abs(l - l0) <= tol * (1 + np.abs(l0)))


def test_loop9_monolithic_matches_library_softmax():
    # the reference schedule against scipy's logsumexp on each gathered path
    Q, dense, shape = _loop9_dense(7)
    scale = 1.0 / math.sqrt(shape["d_qk"])
    o0, l0 = prefix_tree.monolithic(Q, dense, scale)
    for r in range(shape["B"]):
        K = np.concatenate([dense[i].k for i in prefix_tree.path(dense, r)])
        V = np.concatenate([dense[i].v for i in prefix_tree.path(dense, r)])
        s = scale * (K @ Q[r])
        lse = logsumexp(s)
        assert abs(lse - l0[r]) <= 1e-14
        assert np.allclose(np.exp(s - lse) @ V, o0[r], rtol=0, atol=1e-14)


@pytest.mark.parametrize("threshold", [0, 1, 2, 4])
def test_chunk_attention_threshold_changes_buffer_not_result(threshold):
    # 0x0BD: the threshold only moves chunks between the phases
    Q, dense, shape = _loop9_dense(3)
    scale = 1.0 / math.sqrt(shape["d_qk"])
    o0, _ = prefix_tree.monolithic(Q, dense, scale)
    o, _, n_partial = prefix_tree.chunk_attention(Q, dense, scale, threshold=threshold)
    assert n_partial == sum(c.coverage for c in dense if c.coverage > threshold)
    assert np.all(np.abs(o - o0) <= 1e-15 * (1 + np.abs(o0)))


def test_merge_empty_state_is_identity():
    # 0x0BA: the empty part is a two-sided identity, never exp(-inf - -inf)
    s = (np.array([1.0, -2.0, 0.5]), 0.3, 2.0)
    assert prefix_tree.merge_states(prefix_tree.EMPTY, s) is s
    assert prefix_tree.merge_states(s, prefix_tree.EMPTY) is s
    o, l = prefix_tree.finalize(prefix_tree.EMPTY, 3)
    assert np.all(o == 0) and l == -np.inf


def _paged_tree(chunk_rows, cover, hq, hkv, d, p, seed, dtype=np.float32):
    """A pool holding a prefix tree: chunk c gets its own blocks (a ragged
    chunk leaves the rest of its last block holding NaN), placed at seeded
    shuffled ids.  Returns (q, kc, vc, chunks [n, 4], block_ids)."""
    rng = np.random.default_rng(seed)
    nblk = [oracle.num_blocks(n, p) for n in chunk_rows]
    total = sum(nblk) + 3
    perm = rng.permutation(total).astype(np.int32)
    kc = np.full((total, p, hkv, d), np.nan, np.float32)
    vc = np.full((total, p, hkv, d), np.nan, np.float32)
    ids, chunks, nxt = [], [], 0
    for n, (b, e), nb in zip(chunk_rows, cover, nblk):
        blk = perm[nxt:nxt + nb]
        chunks.append((len(ids), n, b, e))
        ids.extend(blk.tolist())
        nxt += nb
        for t in range(n):
            kc[blk[t // p], t % p] = rng.standard_normal((hkv, d))
            vc[blk[t // p], t % p] = rng.standard_normal((hkv, d))
    B = max(e for _, e in cover)
    q = rng.standard_normal((B, hq, d)).astype(np.float32)
    return q, kc, vc, np.array(chunks, np.int32), np.array(ids, np.int32)


def test_chunk_tree_oracle_matches_dense_monolithic():
    # the paged tree oracle (slot tables over a one-row-block view of the
    # pool) against the dense reference schedule, head by head
    rows, cover = [2, 1, 2, 2, 1, 1, 1], [(0, 4), (0, 2), (2, 4), (0, 1), (1, 2), (2, 3), (3, 4)]
    rows = [r * 3 + 1 for r in rows]  # ragged chunks over 4-row blocks
    q, kc, vc, ch, ids = _paged_tree(rows, cover, hq=4, hkv=2, d=8, p=4, seed=5)
    scale = 1 / math.sqrt(8)
    out, lse = oracle.chunk_tree(q, kc, vc, ch, ids, scale)
    for h in range(4):
        kvh = h // 2
        dense = []
        for (f, n, b, e) in ch:
            slots = [(ids[f + t // 4], t % 4) for t in range(n)]
            dense.append(prefix_tree.Chunk(np.array([kc[s][kvh] for s in slots], np.float64),
                                           np.array([vc[s][kvh] for s in slots], np.float64),
                                           int(b), int(e)))
        o, l = prefix_tree.monolithic(q[:, h].astype(np.float64), dense, scale)
        assert np.allclose(out[:, h], o, rtol=0, atol=1e-13)
        assert np.allclose(lse[:, h], l, rtol=0, atol=1e-13)


def test_chunk_tree_two_levels_equal_shared_prefix_bitwise():
    # a root chunk over every sequence plus one private chunk each is the
    # shared-prefix case: the same rows in the same order, so bit-equal
    sp = wl.shared_prefix_batch(batch=5, prefix_len=48, shared_tail=3, suffix_lo=4, suffix_hi=30,
                                hq=4, hkv=2, d=16, p=16, seed=8)
    kc, vc, npre = _shared_prefix_pools(sp)
    q = wl.to_numpy_storage(sp.q)
    out, lse = oracle.shared_prefix(q, kc, vc, sp.prefix_block_ids, sp.prefix_len,
                                    sp.suffix_tables, sp.suffix_lens, sp.scale)
    ids = list(sp.prefix_block_ids)
    chunks = [(0, sp.prefix_len, 0, sp.num_seqs)]
    for r in range(sp.num_seqs):
        n = int(sp.suffix_lens[r])
        chunks.append((len(ids), n, r, r + 1))
        ids.extend(int(x) for x in sp.suffix_tables[r][:oracle.num_blocks(n, sp.block_size)])
    out2, lse2 = oracle.chunk_tree(q, kc, vc, np.array(chunks), np.array(ids), sp.scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_chunk_tree_private_chunks_equal_paged_decode_bitwise():
    b = wl.tiny_batch()
    kc, vc = _oracle_pool_from_batch(b)
    q = wl.to_numpy_storage(b.q)
    tables, lens = b.block_tables, np.asarray(b.seq_lens)
    out, lse = oracle.paged_decode(q, kc, vc, tables, lens, b.scale)
    ids, chunks = [], []
    for r in range(len(lens)):
        nb = oracle.num_blocks(int(lens[r]), kc.shape[1])
        chunks.append((len(ids), int(lens[r]), r, r + 1))
        ids.extend(int(x) for x in tables[r][:nb])
    out2, lse2 = oracle.chunk_tree(q, kc, vc, np.array(chunks), np.array(ids), b.scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_chunk_tree_invariant_under_chunk_order_and_relabeling():
    rows, cover = [9, 5, 7, 3, 6, 1, 2], [(0, 4), (0, 2), (2, 4), (0, 1), (1, 2), (2, 3), (3, 4)]
    q, kc, vc, ch, ids = _paged_tree(rows, cover, hq=2, hkv=1, d=8, p=4, seed=2)
    out, lse = oracle.chunk_tree(q, kc, vc, ch, ids, 0.3)
    # another order of the chunk list: the same keys per row, summed in
    # another order
    perm = [6, 2, 0, 5, 1, 4, 3]
    out2, lse2 = oracle.chunk_tree(q, kc, vc, ch[perm], ids, 0.3)
    assert np.allclose(out, out2, rtol=0, atol=1e-14) and np.allclose(lse, lse2, rtol=0, atol=1e-14)
    # move every block to another physical id: bit-identical
    nb = kc.shape[0]
    relabel = np.random.default_rng(4).permutation(nb)
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[relabel], vc2[relabel] = kc, vc
    out3, lse3 = oracle.chunk_tree(q, kc2, vc2, ch, relabel[ids].astype(np.int32), 0.3)
    assert np.array_equal(out, out3) and np.array_equal(lse, lse3)


def test_chunk_tree_oracle_rejects_bad_snapshots():
    q, kc, vc, ch, ids = _paged_tree([3, 2], [(0, 2), (1, 2)], hq=1, hkv=1, d=4, p=4, seed=0)
    for bad in ([0, 0, 0, 2], [0, 3, 1, 1], [0, 3, 0, 3], [0, 3, -1, 1], [5, 3, 0, 2]):
        c2 = ch.copy()
        c2[0] = bad
        with pytest.raises(ValueError):
            oracle.chunk_tree(q, kc, vc, c2, ids, 1.0)
    ids2 = ids.copy()
    ids2[0] = kc.shape[0]
    with pytest.raises(ValueError):
        oracle.chunk_tree(q, kc, vc, ch, ids2, 1.0)


def test_loop10_shared_work_ledger():
    row = next(r for r in _rows("ledgers.txt") if r[0] == "loop10")
    prefix = int(row[2])
    i = row.index("suffixes")
    j = row.index("logical")
    suffixes = [int(x) for x in row[i + 1:j]]
    logical, unique, saved = int(row[j + 1]), int(row[row.index("unique") + 1]), int(row[-1])
    for p in (16, 32, 64):
        npre = prefix // p
        nxt = npre
        tables, lens = [], []
        for u in suffixes:
            own = list(range(nxt, nxt + oracle.num_blocks(u, p)))
            nxt += len(own)
            tables.append(list(range(npre)) + own)
            lens.append(prefix + u)
        width = max(len(t) for t in tables)
        bt = np.array([t + [-1] * (width - len(t)) for t in tables], np.int32)
        lo, un = oracle.row_ledger(bt, np.array(lens, np.int32), nxt, p)
        assert (lo, un, lo - un) == (logical, unique, saved)


# ------------------------------------------------------------------ MXFP8 pools
def test_e4m3_decode_table():
    # every code against torch's float8_e4m3fn, and the format's closed forms
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_decode(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[~np.isnan(got)], ref[~np.isnan(ref)])
    assert oracle.e4m3_decode(0x38) == 1.0 and oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9 and oracle.e4m3_decode(0x08) == 2.0 ** -6
    assert oracle.e4m3_decode(0x07) == 7 * 2.0 ** -9 and oracle.e4m3_decode(0xB8) == -1.0
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))


def test_e4m3_encode_matches_search_and_library():
    # nearest code, ties to even: the arithmetic encoder against a search over
    # every finite code, and against torch's conversion (which overflows to NaN
    # past 464, where the encoder saturates instead)
    bits = (np.arange(0, 0x7F80, 5, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)
    x = np.concatenate([bits, -bits[::3]])
    fast = np.array([oracle.e4m3_encode(v) for v in x])
    search = np.array([oracle.e4m3_encode_exhaustive(v) for v in x[::4]])
    assert np.array_equal(fast[::4], search)
    m = np.abs(x) <= 464
    lib = torch.tensor(x[m]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fast[m], lib)


def test_e4m3_ties_and_saturation():
    vals = [oracle.e4m3_decode(c) for c in range(0x7F)]
    for c in range(0x7E):  # the midpoint of neighbours goes to the even code
        mid = (vals[c] + vals[c + 1]) / 2
        assert oracle.e4m3_encode(mid) == (c if c % 2 == 0 else c + 1)
    for big in (448.0, 463.99, 464.0, 465.0, 1e9):
        assert oracle.e4m3_encode(big) == 0x7E and oracle.e4m3_encode(-big) == 0xFE
    assert oracle.e4m3_encode(2.0 ** -10) == 0 and oracle.e4m3_encode(3 * 2.0 ** -10) == 2


def test_mx_scale_is_the_smallest_power_that_fits():
    rng = np.random.default_rng(3)
    amax = np.concatenate([np.exp(rng.uniform(-80, 80, 500)), 448.0 * 2.0 ** np.arange(-60, 60)])
    for a in amax:
        s = oracle.mx_scale(a)
        assert 0 < s <= 254
        assert a <= 448.0 * 2.0 ** (s - 127) and a > 448.0 * 2.0 ** (s - 128)
    assert oracle.mx_scale(0.0) == 0


def _mx_shape():
    return (6, 16, 2, 64)


def test_mxfp8_append_layout_and_roundtrip():
    shape = _mx_shape()
    nb, p, hkv, d = shape
    rng = np.random.default_rng(9)
    n = 5
    # group g of every row: E4M3 values times 2^k with the group's largest
    # magnitude 448 * 2^k, so the scale is 2^k and the round trip is exact
    codes = rng.integers(0, 0x7E, size=(n, hkv, d))
    codes[:, :, ::32] = 0x7E
    vals = np.array([[[oracle.e4m3_decode(c) for c in row] for row in head] for head in codes])
    ks = rng.integers(-20, 20, size=(n, hkv, d // 32))
    x = (vals * np.repeat(2.0 ** ks, 32, axis=2)).astype(np.float32)
    kc = np.full(oracle.mxfp8_pool_bytes(*shape), 0xFF, np.uint8)
    vc = kc.copy()
    slots = np.array([0, 17, 33, -1, 95], np.int64)
    assert oracle.kv_append_mxfp8(kc, vc, shape, x, x, slots) == oracle.OK
    plane = nb * p * hkv * d
    for i, s in enumerate(slots):
        if s < 0:
            continue
        b, o = divmod(int(s), p)
        for h in range(hkv):
            el = kc[((b * p + o) * hkv + h) * d:((b * p + o) * hkv + h + 1) * d]
            assert np.array_equal(el, codes[i, h].astype(np.uint8))
            sc = kc[plane + ((b * hkv + h) * p + o) * (d // 32):][:d // 32]
            assert np.array_equal(sc.astype(int) - 127, ks[i, h])
    deq = oracle.mxfp8_to_f32(kc, shape).reshape(nb * p, hkv, d)
    for i, s in enumerate(slots):
        if s >= 0:
            assert np.array_equal(deq[s], x[i])
    # untouched slots keep their bytes (0xFF: NaN codes)
    assert np.isnan(deq[1]).all()


def test_mxfp8_append_error_bound_and_no_saturation():
    shape = (4, 16, 1, 128)
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((10, 1, 128)) * np.exp(rng.uniform(-5, 5, (10, 1, 1)))).astype(np.float32)
    kc = np.zeros(oracle.mxfp8_pool_bytes(*shape), np.uint8)
    vc = kc.copy()
    assert oracle.kv_append_mxfp8(kc, vc, shape, x, x, np.arange(10)) == oracle.OK
    deq = oracle.mxfp8_to_f32(kc, shape).reshape(-1, 1, 128)[:10]
    g = x.reshape(10, 4, 32).astype(np.float64)
    q = deq.reshape(10, 4, 32).astype(np.float64)
    X = 2.0 ** (kc[4 * 16 * 128:][:40].reshape(10, 4).astype(int) - 127)
    scaled = np.abs(g) / X[:, :, None]
    assert scaled.max() <= 448 and (scaled.max(axis=2) > 224).all()  # fits, and the smallest scale
    # nearest-code error: at most half a step of 2^(floor(log2|v|) - 3), or of 2^-9 below 2^-6
    step = np.where(scaled >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(scaled, 1e-300))) - 3),
                    2.0 ** -9)
    assert (np.abs(q / X[:, :, None] - g / X[:, :, None]) <= step / 2 + 1e-12).all()
