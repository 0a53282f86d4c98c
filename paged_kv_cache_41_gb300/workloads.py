"""Seeded synthetic inputs for paged attention decode.

This module only draws inputs: sequence lengths, the order in which the host
block pool hands out physical blocks, and N(0, 1) query/key/value rows.  It
holds none of the attention arithmetic; slot ids come from the host pool
(``pool.py``) and are meant for the device path only (the CPU oracle derives
its own).  Random rows are drawn with a ``torch.Generator`` on the requested
device, so one run always feeds the same values to both sides.

Workloads (sizes from the problem statement):

* ``tiny``: fp32, lengths {35, 100, 16, 1}, block size 16, 4 query / 2 KV
  heads, head_dim 64, 32 pool blocks handed out in a seeded permutation.
* ``llama``: bf16, batch 64, 32/8 heads, head_dim 128, block size 16, lengths
  uniform in [512, 8192], pool = 1.25 x total need, shuffled free FIFO.
* ``long``: bf16, batch 8, lengths uniform in [32768, 65536], 32/8 heads,
  head_dim 128, block size 16 or 64, shuffled placement.
* ``churn``: 256 concurrent requests over 200 steps (see :class:`ChurnTrace`).
* ``shared``: 128 requests on one 2048-token prefix (see :func:`shared_prefix_batch`).
* ``tree``: a prefix tree of several sharing levels (see :func:`prefix_tree_batch`).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

from .pool import BlockPool

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def randn(shape, dtype: str, gen: torch.Generator, device) -> torch.Tensor:
    """N(0, 1) rows, drawn in fp32 and rounded to the storage dtype."""
    x = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    return x.to(DTYPES[dtype])


def make_generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(seed)
    return g


def to_numpy_storage(t: torch.Tensor) -> np.ndarray:
    """Host copy in oracle storage form: float32, or uint16 bits for bf16."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(t.dtype)


@dataclass
class PagedBatch:
    """A decode batch: each sequence's history minus its last token is the
    prefill, the last token is this step's append, then one decode."""
    name: str
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    seq_lens: np.ndarray          # int32 [B], lengths after this step's append
    block_tables: np.ndarray      # int32 [B, max_blocks], -1 padded
    hist_offsets: np.ndarray      # int64 [B + 1], row offsets into k_hist/v_hist
    k_hist: torch.Tensor          # [sum T, Hkv, D] logical K rows, sequence order
    v_hist: torch.Tensor
    q: torch.Tensor               # [B, Hq, D]
    slots: np.ndarray             # int64 [sum T], slot of every history row (host pool)
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return len(self.seq_lens)

    @property
    def max_blocks(self) -> int:
        return self.block_tables.shape[1]

    def last_rows(self) -> np.ndarray:
        """Row index of each sequence's last token (the step's append)."""
        return (self.hist_offsets[1:] - 1).astype(np.int64)

    def prefill_rows(self) -> np.ndarray:
        keep = np.ones(int(self.hist_offsets[-1]), dtype=bool)
        last = self.last_rows()
        keep[last[self.seq_lens > 0]] = False
        return np.nonzero(keep)[0].astype(np.int64)


def _paged_batch(name, dtype, seq_lens, hq, hkv, d, p, num_blocks, seed, device,
                 shuffle=True, scale=None) -> PagedBatch:
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    pool = BlockPool(num_blocks, p, seed=seed, shuffle=shuffle)
    seqs = [pool.new_seq() for _ in seq_lens]
    slot_parts = []
    # prefill every sequence in order, then each sequence's last token
    for s, t in zip(seqs, seq_lens):
        sl, cow = s.append(max(int(t) - 1, 0))
        assert len(cow) == 0
        slot_parts.append([sl])
    for r, (s, t) in enumerate(zip(seqs, seq_lens)):
        if t > 0:
            sl, cow = s.append(1)
            assert len(cow) == 0
            slot_parts[r].append(sl)
    slots = np.concatenate([np.concatenate(x) for x in slot_parts]) if len(seq_lens) else \
        np.zeros(0, np.int64)
    tables, lens = pool.block_tables(seqs)
    assert np.array_equal(lens, seq_lens)
    offs = np.zeros(len(seq_lens) + 1, dtype=np.int64)
    offs[1:] = np.cumsum(seq_lens.astype(np.int64))
    g = make_generator(seed, device)
    total = int(offs[-1])
    k_hist = randn((total, hkv, d), dtype, g, device)
    v_hist = randn((total, hkv, d), dtype, g, device)
    q = randn((len(seq_lens), hq, d), dtype, g, device)
    for s in seqs:
        s.release()
    return PagedBatch(name=name, dtype=dtype, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                      block_size=p, num_blocks=num_blocks,
                      scale=scale if scale is not None else 1.0 / math.sqrt(d),
                      seq_lens=seq_lens, block_tables=tables, hist_offsets=offs,
                      k_hist=k_hist, v_hist=v_hist, q=q, slots=slots, seed=seed)


def pool_size(seq_lens, block_size, factor=1.25) -> int:
    need = sum((int(t) + block_size - 1) // block_size for t in seq_lens)
    return max(1, int(math.ceil(factor * need)))


def tiny_batch(device="cpu", seed=1) -> PagedBatch:
    """fp32; lengths {35, 100, 16, 1}; P=16; Hq=4, Hkv=2, D=64; 32 pool blocks."""
    return _paged_batch("tiny", "f32", [35, 100, 16, 1], 4, 2, 64, 16, 32, seed, device,
                        scale=1.0 / 8.0)


def llama_batch(device="cpu", seed=2, batch=64) -> PagedBatch:
    """bf16; batch 64; Hq=32, Hkv=8, D=128; P=16; lengths uniform in [512, 8192]."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(512, 8192, size=batch, endpoint=True)
    return _paged_batch("llama", "bf16", lens, 32, 8, 128, 16, pool_size(lens, 16), seed, device)


def long_batch(device="cpu", seed=3, block_size=16, batch=8) -> PagedBatch:
    """bf16; batch 8; lengths uniform in [32768, 65536]; Hq=32, Hkv=8, D=128."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(32768, 65536, size=batch, endpoint=True)
    return _paged_batch(f"long_bs{block_size}", "bf16", lens, 32, 8, 128, block_size,
                        pool_size(lens, block_size), seed, device)


def custom_batch(seq_lens, *, dtype="bf16", hq=32, hkv=8, d=128, p=16, num_blocks=None,
                 seed=0, device="cpu", shuffle=True, scale=None) -> PagedBatch:
    if num_blocks is None:
        num_blocks = pool_size(seq_lens, p)
    return _paged_batch("custom", dtype, seq_lens, hq, hkv, d, p, num_blocks, seed, device,
                        shuffle=shuffle, scale=scale)


# --------------------------------------------------------------- shared prefix
@dataclass
class SharedPrefixBatch:
    """Requests forked from one parent whose context is the shared prefix plus
    ``shared_tail`` tokens in a partially filled block.  Each child's first
    append copies that tail block on write (host pool decision) before writing
    its own rows."""
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    prefix_len: int
    shared_tail: int
    parent_table: np.ndarray       # int32 [n_parent_blocks]
    parent_k: torch.Tensor         # [prefix_len + shared_tail, Hkv, D]
    parent_v: torch.Tensor
    parent_slots: np.ndarray       # int64, host pool slots of the parent rows
    prefix_block_ids: np.ndarray   # int32 [prefix_len / P]
    suffix_lens: np.ndarray        # int32 [B], includes the shared tail rows
    suffix_tables: np.ndarray      # int32 [B, max_suffix_blocks]
    cow_pairs: np.ndarray          # int64 [n_cow, 2]
    child_offsets: np.ndarray      # int64 [B + 1] into child_k/child_v
    child_k: torch.Tensor          # private rows of every child, in order
    child_v: torch.Tensor
    child_slots: np.ndarray        # int64, host pool slots of the private rows
    q: torch.Tensor                # [B, Hq, D]

    @property
    def num_seqs(self) -> int:
        return len(self.suffix_lens)


def shared_prefix_batch(device="cpu", seed=5, batch=128, prefix_len=2048, shared_tail=8,
                        suffix_lo=16, suffix_hi=512, hq=32, hkv=8, d=128, p=16,
                        dtype="bf16") -> SharedPrefixBatch:
    rng = np.random.default_rng(seed)
    suffix = rng.integers(suffix_lo, suffix_hi, size=batch, endpoint=True).astype(np.int32)
    assert prefix_len % p == 0 and 0 <= shared_tail < p and (suffix >= shared_tail).all()
    need = (prefix_len + p - 1) // p + 1 + sum((int(u) + p - 1) // p for u in suffix)
    nb = int(math.ceil(1.25 * need))
    pool = BlockPool(nb, p, seed=seed, shuffle=True)
    parent = pool.new_seq()
    parent_slots, cow = parent.append(prefix_len + shared_tail)
    assert len(cow) == 0
    parent_table = parent.blocks()
    children = [parent.fork() for _ in range(batch)]
    parent.release()
    cows, child_slots = [], []
    for c, u in zip(children, suffix):
        sl, cw = c.append(int(u) - shared_tail)
        child_slots.append(sl)
        if len(cw):
            cows.append(cw)
    npre = prefix_len // p
    max_suf = max(c.num_blocks for c in children) - npre
    tables, lens = pool.block_tables(children, max_blocks=npre + max_suf)
    prefix_ids = tables[0, :npre].copy()
    assert (tables[:, :npre] == prefix_ids).all()
    g = make_generator(seed, device)
    parent_k = randn((prefix_len + shared_tail, hkv, d), dtype, g, device)
    parent_v = randn((prefix_len + shared_tail, hkv, d), dtype, g, device)
    offs = np.zeros(batch + 1, dtype=np.int64)
    offs[1:] = np.cumsum(suffix.astype(np.int64) - shared_tail)
    child_k = randn((int(offs[-1]), hkv, d), dtype, g, device)
    child_v = randn((int(offs[-1]), hkv, d), dtype, g, device)
    q = randn((batch, hq, d), dtype, g, device)
    for c in children:
        c.release()
    return SharedPrefixBatch(
        dtype=dtype, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=p, num_blocks=nb,
        scale=1.0 / math.sqrt(d), prefix_len=prefix_len, shared_tail=shared_tail,
        parent_table=parent_table, parent_k=parent_k, parent_v=parent_v,
        parent_slots=parent_slots, prefix_block_ids=prefix_ids, suffix_lens=suffix,
        suffix_tables=np.ascontiguousarray(tables[:, npre:]),
        cow_pairs=np.concatenate(cows).astype(np.int64) if cows else np.zeros((0, 2), np.int64),
        child_offsets=offs, child_k=child_k, child_v=child_v,
        child_slots=np.concatenate(child_slots) if child_slots else np.zeros(0, np.int64), q=q)


# --------------------------------------------------------------- prefix tree
@dataclass
class PrefixTreeBatch:
    """A tree snapshot in a paged pool: ``chunks`` rows are (first id, rows,
    seq begin, seq end) in tree order (parents first); chunk c's rows live in
    blocks block_ids[first id ...] handed out by the host pool, one chunk per
    pool sequence (a ragged chunk leaves the rest of its last block unused).
    Chunk rows are drawn in chunk order into k_rows / v_rows; ``slots`` is
    their host-pool slot, for the device path only."""
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    chunks: np.ndarray             # int32 [n, 4]
    block_ids: np.ndarray          # int32 [sum of blocks]
    row_offsets: np.ndarray        # int64 [n + 1] into k_rows / v_rows
    k_rows: torch.Tensor           # [sum of rows, Hkv, D]
    v_rows: torch.Tensor
    slots: np.ndarray              # int64 [sum of rows]
    q: torch.Tensor                # [B, Hq, D]

    @property
    def num_seqs(self) -> int:
        return self.q.shape[0]


def multi_level_tree(batch, root_len, groups, group_len, leaf_lo, leaf_hi, seed):
    """(rows, begin, end) of a three-level tree: one root chunk over every
    sequence, ``groups`` equal groups of consecutive sequences each with its
    own chunk, and one private leaf per sequence of U{leaf_lo..leaf_hi}
    rows.  Group chunk lengths are drawn in [group_len / 2, group_len]."""
    rng = np.random.default_rng(seed)
    tree = [(root_len, 0, batch)]
    per = batch // groups
    for g in range(groups):
        lo, hi = g * per, batch if g == groups - 1 else (g + 1) * per
        tree.append((int(rng.integers(group_len // 2, group_len, endpoint=True)), lo, hi))
    leaves = rng.integers(leaf_lo, leaf_hi, size=batch, endpoint=True)
    tree.extend((int(n), r, r + 1) for r, n in enumerate(leaves))
    return tree


def prefix_tree_batch(tree, device="cpu", seed=7, hq=32, hkv=8, d=128, p=16, dtype="bf16",
                      batch=None) -> PrefixTreeBatch:
    """Place the chunks of ``tree`` ((rows, begin, end) in tree order) in a
    shuffled pool of 1.25 x the blocks they need and draw N(0, 1) rows."""
    nblk = [(n + p - 1) // p for n, _, _ in tree]
    nb = max(1, int(math.ceil(1.25 * sum(nblk))))
    pool = BlockPool(nb, p, seed=seed, shuffle=True)
    chunks, ids, slots, offs = [], [], [], [0]
    for (n, b, e) in tree:
        s = pool.new_seq()
        sl, cow = s.append(n)
        assert len(cow) == 0
        chunks.append((len(ids), n, b, e))
        ids.extend(int(x) for x in s.blocks())
        slots.append(sl)
        offs.append(offs[-1] + n)
    B = batch if batch is not None else max(e for _, _, e in tree)
    g = make_generator(seed, device)
    total = offs[-1]
    k_rows = randn((total, hkv, d), dtype, g, device)
    v_rows = randn((total, hkv, d), dtype, g, device)
    q = randn((B, hq, d), dtype, g, device)
    return PrefixTreeBatch(
        dtype=dtype, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=p, num_blocks=nb,
        scale=1.0 / math.sqrt(d), chunks=np.array(chunks, np.int32).reshape(-1, 4),
        block_ids=np.array(ids, np.int32), row_offsets=np.array(offs, np.int64), k_rows=k_rows,
        v_rows=v_rows, slots=np.concatenate(slots).astype(np.int64) if slots else
        np.zeros(0, np.int64), q=q)


# --------------------------------------------------------------- churn trace
@dataclass
class ChurnStep:
    """Everything one step of the churn trace hands the device."""
    arrival_rows: int              # prompt rows appended this step (not decode)
    arrival_slots: np.ndarray      # int64 host pool slots for those rows
    step_slots: np.ndarray         # int64 [B] slot of each active request's new token
    block_tables: np.ndarray       # int32 [B, max_blocks]
    seq_lens: np.ndarray           # int32 [B]
    arrival_seq_index: np.ndarray  # int32, which batch row each arrival row belongs to
    arrival_positions: np.ndarray  # int64, logical position of each arrival row


class ChurnTrace:
    """256 concurrent requests over 200 decode steps.

    Prompt lengths are lognormal (median 1024, sigma 1.0, capped at 16384),
    output lengths geometric with mean 200.  A finished request releases its
    blocks to the FIFO tail; the arrival replacing it takes blocks from the
    head.  The pool holds 1.25 x the peak live blocks of a dry run of the
    same seeded trace.  Every step appends one token per active request,
    then decodes.
    """

    def __init__(self, seed=4, concurrency=256, steps=200, block_size=16, median=1024,
                 sigma=1.0, cap=16384, mean_out=200, num_blocks=None):
        self.seed, self.concurrency, self.steps, self.block_size = seed, concurrency, steps, block_size
        rng = np.random.default_rng(seed)
        n_req = concurrency * 8 + 64
        prompts = np.exp(np.log(median) + sigma * rng.standard_normal(n_req))
        self.prompts = np.clip(np.rint(prompts), 1, cap).astype(np.int64)
        self.outputs = rng.geometric(1.0 / mean_out, size=n_req).astype(np.int64)
        if num_blocks is None:
            peak = self._dry_run()
            num_blocks = int(math.ceil(1.25 * peak))
        self.num_blocks = num_blocks

    def _dry_run(self) -> int:
        p = self.block_size
        live = []
        nxt = 0
        peak = 0
        lens, left = [], []
        for _ in range(self.concurrency):
            lens.append(int(self.prompts[nxt]))
            left.append(int(self.outputs[nxt]))
            nxt += 1
        for _ in range(self.steps):
            for i in range(self.concurrency):
                lens[i] += 1
            peak = max(peak, sum((t + p - 1) // p for t in lens))
            for i in range(self.concurrency):
                left[i] -= 1
                if left[i] == 0:
                    lens[i] = int(self.prompts[nxt])
                    left[i] = int(self.outputs[nxt])
                    nxt += 1
        del live
        return peak

    def run(self):
        """Yields ChurnStep objects; the pool state advances as they are consumed."""
        p = self.block_size
        pool = BlockPool(self.num_blocks, p, seed=self.seed, shuffle=True)
        seqs, left = [], []
        nxt = 0
        pending_slots, pending_seq, pending_pos = [], [], []
        for i in range(self.concurrency):
            s = pool.new_seq()
            sl, _ = s.append(int(self.prompts[nxt]))
            pending_slots.append(sl)
            pending_seq.append(np.full(len(sl), i, np.int32))
            pending_pos.append(np.arange(len(sl), dtype=np.int64))
            seqs.append(s)
            left.append(int(self.outputs[nxt]))
            nxt += 1
        max_blocks = (int(self.prompts.max()) + self.steps + p) // p + 1
        for _ in range(self.steps):
            step_slots = np.empty(self.concurrency, np.int64)
            for i, s in enumerate(seqs):
                sl, cow = s.append(1)
                assert len(cow) == 0
                step_slots[i] = sl[0]
            tables, lens = pool.block_tables(seqs, max_blocks=max_blocks)
            arr_slots = np.concatenate(pending_slots) if pending_slots else np.zeros(0, np.int64)
            yield ChurnStep(arrival_rows=len(arr_slots), arrival_slots=arr_slots,
                            step_slots=step_slots, block_tables=tables, seq_lens=lens,
                            arrival_seq_index=np.concatenate(pending_seq) if pending_seq
                            else np.zeros(0, np.int32),
                            arrival_positions=np.concatenate(pending_pos) if pending_pos
                            else np.zeros(0, np.int64))
            pending_slots, pending_seq, pending_pos = [], [], []
            for i in range(self.concurrency):
                left[i] -= 1
                if left[i] == 0:
                    seqs[i].release()
                    s = pool.new_seq()
                    sl, _ = s.append(int(self.prompts[nxt]))
                    pending_slots.append(sl)
                    pending_seq.append(np.full(len(sl), i, np.int32))
                    pending_pos.append(np.arange(len(sl), dtype=np.int64))
                    seqs[i] = s
                    left[i] = int(self.outputs[nxt])
                    nxt += 1
        for s in seqs:
            s.release()
