"""Host block pool: FIFO order, refcounts, the three append paths, tables.

The slot mapping the pool produces for the device path is compared with the
CPU oracle's own translation of the same block tables.
"""
import numpy as np
import pytest

import oracle
from paged_kv_cache_41_gb300.pool import BlockPool, PoolExhausted


def test_fifo_order_unshuffled_and_tail_push():
    pool = BlockPool(4, 16, shuffle=False)
    assert [pool.alloc() for _ in range(3)] == [0, 1, 2]
    pool.decref(1)
    assert pool.alloc() == 3          # head of the FIFO first
    assert pool.alloc() == 1          # the freed id went to the tail
    with pytest.raises(PoolExhausted):
        pool.alloc()


def test_seeded_shuffle_is_a_permutation_and_reproducible():
    a = BlockPool(32, 16, seed=1)
    b = BlockPool(32, 16, seed=1)
    c = BlockPool(32, 16, seed=2)
    ia = [a.alloc() for _ in range(32)]
    ib = [b.alloc() for _ in range(32)]
    ic = [c.alloc() for _ in range(32)]
    assert sorted(ia) == list(range(32)) and ia == ib and ia != ic


def test_refcount_conservation_under_fork_and_release():
    pool = BlockPool(64, 16, seed=3)
    s = pool.new_seq()
    s.append(40)                      # 3 blocks
    kids = [s.fork() for _ in range(3)]
    for b in s.blocks():
        assert pool.refcount(int(b)) == 4
    s.release()
    for k in kids:
        k.release()
    assert pool.num_free == 64        # N_pool = N_free + N_live with nothing live


def test_append_paths_new_block_private_tail_cow():
    pool = BlockPool(16, 16, seed=4)
    s = pool.new_seq()
    slots, cow = s.append(20)         # offsets 0 -> new blocks; 2 blocks
    assert s.num_blocks == 2 and len(cow) == 0
    slots2, cow = s.append(1)         # private tail: write in place at offset 4
    assert len(cow) == 0 and slots2[0] == s.blocks()[1] * 16 + 4
    child = s.fork()
    tail = int(s.blocks()[1])
    slots3, cow = child.append(1)     # shared tail with free slots: copy on write
    assert cow.shape == (1, 2) and cow[0, 0] == tail and cow[0, 1] == child.blocks()[1]
    assert pool.refcount(tail) == 1 and pool.refcount(int(cow[0, 1])) == 1
    assert slots3[0] == cow[0, 1] * 16 + 5
    slots4, cow = s.append(1)         # the parent is the unique owner again
    assert len(cow) == 0 and slots4[0] == tail * 16 + 5


def test_full_shared_tail_needs_no_copy():
    pool = BlockPool(8, 16, seed=5)
    s = pool.new_seq()
    s.append(32)
    child = s.fork()
    _, cow = child.append(1)          # offset 0: a new block, nothing copied
    assert len(cow) == 0 and child.num_blocks == 3


def test_exhaustion_leaves_state_unchanged():
    pool = BlockPool(2, 16, seed=6)
    s = pool.new_seq()
    s.append(20)
    with pytest.raises(PoolExhausted):
        s.append(20)
    assert s.length == 20 and pool.num_free == 0


def test_pool_slots_equal_oracle_translation_of_tables():
    pool = BlockPool(200, 16, seed=7)
    seqs = [pool.new_seq() for _ in range(5)]
    lens = [35, 100, 16, 1, 257]
    all_slots = [s.append(t)[0] for s, t in zip(seqs, lens)]
    tables, got_lens = pool.block_tables(seqs)
    assert list(got_lens) == lens
    for r, (t, sl) in enumerate(zip(lens, all_slots)):
        want = [oracle.slot_for_position(tables[r], 16, i) for i in range(t)]
        assert list(sl) == want
        assert (tables[r, oracle.num_blocks(t, 16):] == -1).all()


def test_block_tables_reject_narrow_width():
    pool = BlockPool(8, 16, seed=8)
    s = pool.new_seq()
    s.append(40)
    with pytest.raises(ValueError):
        pool.block_tables([s], max_blocks=2)
