"""Host logic of the prefix-tree planner (pkv_chunk_tree_plan), without a GPU.

The plan is opaque to callers; these tests read its header and sections with
the layout pkv_api.cu writes, to check the planner's bookkeeping against
counts derived here from the tree itself: which chunks go chunk-first, the
padded partial rows, the work items covering every (chunk, query-tile pair,
key) exactly once, the sequence-first segments, and each sequence's state
list in tree order.
"""
import ctypes
import struct

import numpy as np
import pytest
import torch

from paged_kv_cache_41_gb300 import build, pkv

HDR = struct.Struct("<IIq4i2i6iq8Q3Q4Q")
FIELDS = ("magic version num_blocks block_size num_kv_heads head_dim dtype num_seqs num_q_heads "
          "n_items s_max cf_rows n_pseudo pseudo_max_blocks n_states decode_ctas items_off "
          "cf_ids_off ptab_off plen_off pq_off seqptr_off states_off plan_bytes ws_lse_off "
          "ws_dec_off ws_bytes dec_pre_off dec_lse_off dec_o_off dec_total").split()


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build_all()


def _cache(nb=64, p=16, hkv=2, d=64, dtype=torch.bfloat16):
    return torch.empty(nb, p, hkv, d, dtype=dtype)  # shape only: planning reads no data


def _plan(k, chunks, ids, b, hq, threshold=-1):
    plan = pkv.chunk_tree_plan(k, chunks, ids, b, hq, threshold, device="cpu")
    raw = plan.host.numpy().tobytes()
    h = dict(zip(FIELDS, HDR.unpack_from(raw)))
    assert h["magic"] == 0x54564B50 and h["plan_bytes"] == len(raw)

    def arr(off, n, dt=np.int32):
        return np.frombuffer(raw, dt, count=n, offset=off)

    h["items"] = arr(h["items_off"], 8 * h["n_items"]).reshape(-1, 8)
    h["seq_ptr"] = arr(h["seqptr_off"], b + 1)
    h["states"] = arr(h["states_off"], 2 * h["n_states"], np.int64).reshape(-1, 2)
    h["plen"] = arr(h["plen_off"], h["n_pseudo"])
    h["pq"] = arr(h["pq_off"], h["n_pseudo"])
    h["ptab"] = arr(h["ptab_off"], h["n_pseudo"] * h["pseudo_max_blocks"]).reshape(
        h["n_pseudo"], h["pseudo_max_blocks"])
    return plan, h


LOOP9 = [(2, 0, 4), (1, 0, 2), (2, 2, 4), (2, 0, 1), (1, 1, 2), (1, 2, 3), (1, 3, 4)]


def _cf_at(tree, cf, p=16):
    """(offset among the chunk-first chunks' ids, chunk) for each chunk-first chunk."""
    out, nxt = [], 0
    for c in cf:
        out.append((nxt, c))
        nxt += -(-tree[c][0] // p)
    return out


def _chunks(tree, p):
    out, nxt = [], 0
    for n, b, e in tree:
        out.append((nxt, n, b, e))
        nxt += -(-n // p)
    return np.array(out, np.int32), np.arange(nxt, dtype=np.int32)


@pytest.mark.parametrize("threshold,cf", [(-1, [0, 1, 2]), (0, list(range(7))), (1, [0, 1, 2]),
                                          (2, [0]), (4, [])])
def test_loop9_phases_follow_the_threshold(threshold, cf):
    # 0x0BD: chunks covering more than the threshold go chunk-first
    tree = [(n * 40 + 3, b, e) for n, b, e in LOOP9]
    ch, ids = _chunks(tree, 16)
    _, h = _plan(_cache(), ch, ids, 4, 8, threshold)  # G = 4: 32 requests per query tile
    cov = [e - b for _, b, e in tree]
    assert h["cf_rows"] == 32 * len(cf)  # each chunk-first chunk pads to one query tile
    assert h["n_pseudo"] == sum(c for i, c in enumerate(cov) if i not in cf)
    # one state per (sequence, chunk on its path), times the chunk-first
    # chunks' key splits
    splits = {c: len({it[6] for it in h["items"] if it[0] == off}) for off, c in _cf_at(tree, cf)}
    per_seq = [sum(splits.get(i, 1) for i, (_, b, e) in enumerate(tree) if b <= r < e)
               for r in range(4)]
    assert h["seq_ptr"].tolist() == np.concatenate([[0], np.cumsum(per_seq)]).tolist()
    assert h["n_states"] == sum(per_seq)
    # every (chunk-first chunk, key) is covered by exactly one item (one pair
    # here); items name a chunk by where its ids start among the chunk-first
    # chunks' ids
    at = dict(_cf_at(tree, cf))
    keys = {}
    for it in h["items"]:
        ids_off, key0, nkeys, req0, nreq, st_req0, split = it[:7]
        c = at[ids_off]
        assert req0 == tree[c][1] and nreq == cov[c] and st_req0 == 32 * cf.index(c)
        for k in range(key0, key0 + nkeys):
            assert (c, k) not in keys
            keys[(c, k)] = split
    assert sorted(keys) == sorted((c, k) for c in cf for k in range(tree[c][0]))


def test_entries_list_each_path_in_tree_order():
    tree = [(200, 0, 6), (50, 0, 3), (70, 3, 6)] + [(5 + r, r, r + 1) for r in range(6)]
    ch, ids = _chunks(tree, 16)
    _, h = _plan(_cache(), ch, ids, 6, 8, 1)
    cf_rows = h["cf_rows"]
    assert cf_rows == 3 * 32 and h["n_pseudo"] == 6
    S, Hq = h["s_max"], 8
    for r in range(6):
        refs = h["states"][h["seq_ptr"][r]:h["seq_ptr"][r + 1]].tolist()
        # root's key splits (row r), the group's (rows 32.. or 64..), then the
        # private leaf as one decode segment after every chunk-first state
        grp_row = 32 + r if r < 3 else 64 + r - 3
        root = [[r * Hq * S + s, S] for s in range(S)]
        assert refs[:S] == root
        grp = refs[S:-1]
        assert 1 <= len(grp) <= S and grp == [[grp_row * Hq * S + s, S] for s in range(len(grp))]
        assert refs[-1] == [cf_rows * Hq * S + r * Hq, 1]
    # the segments carry their sequence, rows and the chunk's blocks
    assert h["pq"].tolist() == list(range(6)) and h["plen"].tolist() == [5, 6, 7, 8, 9, 10]
    for j in range(6):
        f = ch[3 + j][0]
        assert h["ptab"][j][0] == ids[f]


def test_split_count_bounds_the_grid():
    # one long shared chunk: splits multiply until (items x kv heads) would
    # pass one wave of the SMs
    tree = [(4096, 0, 64)] + [(8, r, r + 1) for r in range(64)]
    ch, ids = _chunks(tree, 16)
    _, h = _plan(_cache(nb=4096, hkv=8, d=128), ch, ids, 64, 32, 1)
    n_items, s_max = h["n_items"], h["s_max"]
    assert n_items == s_max * 1  # 64 requests x 4 heads = 2 tiles = one pair
    assert n_items * 8 <= 160 and s_max >= 8
    assert sum(it[2] for it in h["items"]) == 4096


def test_fp32_cache_runs_everything_sequence_first():
    tree = [(40, 0, 4), (3, 0, 1), (3, 1, 2)]
    ch, ids = _chunks(tree, 16)
    _, h = _plan(_cache(dtype=torch.float32), ch, ids, 4, 8, 0)
    assert h["n_items"] == 0 and h["cf_rows"] == 0 and h["n_pseudo"] == 6


def test_workspace_holds_states_and_decode():
    tree = [(300, 0, 8)] + [(10, r, r + 1) for r in range(8)]
    ch, ids = _chunks(tree, 16)
    _, h = _plan(_cache(), ch, ids, 8, 8, 1)
    n_states = h["cf_rows"] * 8 * h["s_max"] + h["n_pseudo"] * 8
    assert h["ws_lse_off"] >= n_states * 64 * 4
    assert h["ws_dec_off"] >= h["ws_lse_off"] + n_states * 4
    assert h["ws_bytes"] == h["ws_dec_off"] + h["dec_total"] and h["dec_total"] > 0


@pytest.mark.parametrize("bad", [
    [(0, 0, 0, 2)],            # empty chunk
    [(0, 3, 1, 1)],            # empty interval
    [(0, 3, 0, 5)],            # interval past the batch
    [(0, 3, -1, 2)],           # negative begin
    [(3, 40, 0, 2)],           # ids past the list
])
def test_planner_rejects_bad_chunks(bad):
    with pytest.raises(pkv.PkvError) as e:
        pkv.chunk_tree_plan(_cache(), np.array(bad, np.int32), np.arange(4, dtype=np.int32), 4, 8,
                            device="cpu")
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG


def test_planner_rejects_block_ids_outside_the_pool():
    with pytest.raises(pkv.PkvError) as e:
        pkv.chunk_tree_plan(_cache(nb=8), np.array([(0, 3, 0, 2)], np.int32),
                            np.array([8], np.int32), 2, 8, device="cpu")
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG


def test_planner_reports_capacity():
    lib = pkv.load_library()
    desc = pkv.cache_desc(_cache())
    ch = np.array([(0, 20, 0, 2), (2, 5, 0, 1)], np.int32)
    ids = np.arange(3, dtype=np.int32)
    pb, wb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    args = (ctypes.byref(desc), ctypes.c_void_p(ch.ctypes.data), 2,
            ctypes.c_void_p(ids.ctypes.data), 3, 2, 8, -1)
    assert lib.pkv_chunk_tree_plan(*args, None, 0, ctypes.byref(pb), ctypes.byref(wb)) == 0
    assert pb.value > 0 and wb.value > 0
    buf = (ctypes.c_ubyte * pb.value)()
    assert lib.pkv_chunk_tree_plan(*args, buf, pb.value - 1, ctypes.byref(pb),
                                   ctypes.byref(wb)) == pkv.PKV_ERR_CAPACITY
    assert lib.pkv_chunk_tree_plan(*args, buf, pb.value, ctypes.byref(pb), ctypes.byref(wb)) == 0
