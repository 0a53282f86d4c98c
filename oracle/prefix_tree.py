"""Prefix-tree attention schedules over dense per-chunk K/V, in binary64.

TEST INFRASTRUCTURE ONLY.  Only the test suite may import this module; the
product library never loads it and shares no code with it.

Follows "M5.3 - KV Memory Layout and Exact Reuse":
  * 0x0BA: a partition of a row's scores gives per-part states; merging them
    by log-sum-exp (never by averaging normalised outputs) is exact, and an
    empty part is the merge's identity;
  * 0x0BB: a tree snapshot is an ordered list of chunks, each with its K/V
    rows and a half-open interval [begin, end) of the sequences it covers; a
    sequence's path is every chunk whose interval holds it, in tree order;
  * 0x0BC (Hydragen): each chunk attends to all the queries it covers at once
    and emits (normalised output, LSE) per query; every sequence then merges
    the states of its path;
  * 0x0BD (ChunkAttention): chunks covering more than ``threshold`` sequences
    are attended first, their unnormalised states (u, m, l) kept in a buffer
    of partial rows; each sequence then walks its path, taking the kept
    state of a shared chunk or attending to a private one itself, and merges
    online;
  * 0x0BE: the three schedules (the monolithic reference, Hydragen,
    ChunkAttention) agree to rounding, and the work and payload ledgers.

A snapshot here is ``(Q, chunks)`` with ``Q`` of shape [B, d_qk] (one head,
one query per sequence) and ``chunks`` a list of ``Chunk``.  Widths d_qk and
d_v may differ, as in the fixture of 0x0BB.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass
class Chunk:
    k: np.ndarray   # [rows, d_qk]
    v: np.ndarray   # [rows, d_v]
    begin: int      # first covered sequence
    end: int        # one past the last covered sequence

    @property
    def rows(self) -> int:
        return self.k.shape[0]

    @property
    def coverage(self) -> int:
        return self.end - self.begin


def path(chunks, r: int) -> list:
    """Indices of the chunks covering sequence r, in tree order (0x0BB)."""
    return [i for i, c in enumerate(chunks) if c.begin <= r < c.end]


def monolithic(Q: np.ndarray, chunks, scale: float):
    """The reference schedule: concatenate each path and run one softmax row
    over it.  Returns (out [B, d_v], lse [B])."""
    B = Q.shape[0]
    d_v = chunks[0].v.shape[1]
    out = np.zeros((B, d_v))
    lse = np.full(B, -np.inf)
    for r in range(B):
        idx = path(chunks, r)
        if not idx:
            continue
        K = np.concatenate([chunks[i].k for i in idx])
        V = np.concatenate([chunks[i].v for i in idx])
        s = scale * (K @ Q[r])
        m = s.max()
        p = np.exp(s - m)
        out[r] = (p @ V) / p.sum()
        lse[r] = m + np.log(p.sum())
    return out, lse


# ------------------------------------------------------------ Hydragen, 0x0BC
def attend_group(Qg: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """All queries of a group against one chunk: (normalised output [n, d_v],
    natural-log LSE [n])."""
    S = scale * (Qg @ K.T)                  # [n, rows]
    m = S.max(axis=1, keepdims=True)
    P = np.exp(S - m)
    l = P.sum(axis=1)
    return (P @ V) / l[:, None], m[:, 0] + np.log(l)


def merge_normalised(outs, lses):
    """Combine (normalised output, LSE) parts of one row by their masses
    exp(LSE - max LSE); the parts' keys are disjoint."""
    lses = np.asarray(lses, dtype=np.float64)
    top = lses.max()
    w = np.exp(lses - top)
    o = sum(wi * oi for wi, oi in zip(w, outs)) / w.sum()
    return o, top + np.log(w.sum())


def hydragen(Q: np.ndarray, chunks, scale: float):
    """Hierarchical Hydragen: one batched attention per chunk over the
    queries it covers, then a per-sequence merge of the path's parts."""
    B = Q.shape[0]
    parts = [[] for _ in range(B)]
    for c in chunks:
        O, L = attend_group(Q[c.begin:c.end], c.k, c.v, scale)
        for j in range(c.coverage):
            parts[c.begin + j].append((O[j], L[j]))
    d_v = chunks[0].v.shape[1]
    out = np.zeros((B, d_v))
    lse = np.full(B, -np.inf)
    for r in range(B):
        if parts[r]:
            out[r], lse[r] = merge_normalised([p[0] for p in parts[r]], [p[1] for p in parts[r]])
    return out, lse


# ------------------------------------------------------- ChunkAttention, 0x0BD
EMPTY = None  # the empty state: identity of the merge, never (0, -inf, 0)


def partial_state(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """Unnormalised online-softmax state (u, m, l) of one query over K/V."""
    s = scale * (K @ q)
    m = s.max()
    p = np.exp(s - m)
    return p @ V, m, p.sum()


def merge_states(a, b):
    """Online-softmax merge of two (u, m, l) states; EMPTY is the identity,
    handled by a branch before any exponent is formed."""
    if a is EMPTY:
        return b
    if b is EMPTY:
        return a
    ua, ma, la = a
    ub, mb, lb = b
    m = max(ma, mb)
    ea, eb = np.exp(ma - m), np.exp(mb - m)
    return ea * ua + eb * ub, m, ea * la + eb * lb


def finalize(state, d_v: int):
    if state is EMPTY:
        return np.zeros(d_v), -np.inf
    u, m, l = state
    return u / l, m + np.log(l)


def chunk_attention(Q: np.ndarray, chunks, scale: float, threshold: int = 1):
    """Two-phase ChunkAttention.  Returns (out [B, d_v], lse [B],
    partial_rows): chunks covering more than ``threshold`` sequences are
    materialised first into partial rows (offset = rows of the earlier shared
    chunks); the sequence-first phase reads them back."""
    B = Q.shape[0]
    d_v = chunks[0].v.shape[1]
    offset = {}
    partial = []
    for i, c in enumerate(chunks):            # chunk-first phase
        if c.coverage <= threshold:
            continue
        offset[i] = len(partial)
        for r in range(c.begin, c.end):
            partial.append(partial_state(Q[r], c.k, c.v, scale))
    out = np.zeros((B, d_v))
    lse = np.full(B, -np.inf)
    for r in range(B):                        # sequence-first phase
        state = EMPTY
        for i in path(chunks, r):
            c = chunks[i]
            if i in offset:
                part = partial[offset[i] + r - c.begin]
            else:
                part = partial_state(Q[r], c.k, c.v, scale)
            state = merge_states(state, part)
        out[r], lse[r] = finalize(state, d_v)
    return out, lse, len(partial)


# -------------------------------------------------------------- ledger, 0x0BE
def ledger(chunks, d_qk: int, d_v: int, elem_bytes: int = 2, state_bytes: int = 4,
           threshold: int = 1) -> dict:
    """Work and payload counts of a snapshot: logical (query, key) pairs,
    unique physical K/V rows, the duplicate reads sharing saves, the K/V
    payloads without and with sharing, and the partial-state buffer of the
    chunk-first phase (output in the element type, max and sum in the state
    type)."""
    logical = sum(c.rows * c.coverage for c in chunks)
    physical = sum(c.rows for c in chunks)
    row = (d_qk + d_v) * elem_bytes
    partial_rows = sum(c.coverage for c in chunks if c.coverage > threshold)
    partial_row = d_v * elem_bytes + 2 * state_bytes
    return {
        "logical_pairs": logical,
        "physical_rows": physical,
        "saved_reads": logical - physical,
        "kv_row_bytes": row,
        "baseline_payload": logical * row,
        "shared_payload": physical * row,
        "partial_rows": partial_rows,
        "partial_row_bytes": partial_row,
        "partial_buffer": partial_rows * partial_row,
    }
