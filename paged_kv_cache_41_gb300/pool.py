"""ctypes binding of the host block pool (``include/pkv_pool.h``).

The pool only generates inputs: block ids, slot mappings, copy-on-write pairs
and dense block tables.  It is plain C; this module marshals arguments.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
POOL_LIB_PATH = os.path.join(_HERE, "libpkv_pool.so")

_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(POOL_LIB_PATH):
            raise RuntimeError(
                f"{POOL_LIB_PATH} is missing: build it with paged_kv_cache_41_gb300.build.build_all()")
        lib = ctypes.CDLL(POOL_LIB_PATH)
        vp, i64, i32, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64
        lib.pkv_pool_create.restype = vp
        lib.pkv_pool_create.argtypes = [i64, i32, u64, ctypes.c_int]
        lib.pkv_pool_destroy.argtypes = [vp]
        lib.pkv_pool_num_blocks.restype = i64
        lib.pkv_pool_num_blocks.argtypes = [vp]
        lib.pkv_pool_block_size.restype = i32
        lib.pkv_pool_block_size.argtypes = [vp]
        lib.pkv_pool_num_free.restype = i64
        lib.pkv_pool_num_free.argtypes = [vp]
        lib.pkv_pool_alloc.restype = i32
        lib.pkv_pool_alloc.argtypes = [vp]
        lib.pkv_pool_refcount.restype = i32
        lib.pkv_pool_refcount.argtypes = [vp, i32]
        lib.pkv_pool_incref.restype = ctypes.c_int
        lib.pkv_pool_incref.argtypes = [vp, i32]
        lib.pkv_pool_decref.restype = ctypes.c_int
        lib.pkv_pool_decref.argtypes = [vp, i32]
        lib.pkv_seq_create.restype = vp
        lib.pkv_seq_create.argtypes = [vp]
        lib.pkv_seq_fork.restype = vp
        lib.pkv_seq_fork.argtypes = [vp, vp]
        lib.pkv_seq_release.argtypes = [vp, vp]
        lib.pkv_seq_len.restype = i64
        lib.pkv_seq_len.argtypes = [vp]
        lib.pkv_seq_num_blocks.restype = i32
        lib.pkv_seq_num_blocks.argtypes = [vp]
        lib.pkv_seq_block.restype = i32
        lib.pkv_seq_block.argtypes = [vp, i32]
        lib.pkv_seq_append_tokens.restype = ctypes.c_int
        lib.pkv_seq_append_tokens.argtypes = [vp, vp, i64, vp, vp, ctypes.POINTER(i32)]
        lib.pkv_build_block_tables.restype = ctypes.c_int
        lib.pkv_build_block_tables.argtypes = [vp, i32, i32, vp, vp]
        _lib = lib
    return _lib


class PoolExhausted(RuntimeError):
    pass


class Seq:
    """One request's block list inside a :class:`BlockPool`."""

    def __init__(self, pool: "BlockPool", handle: int):
        self.pool = pool
        self.handle = handle

    @property
    def length(self) -> int:
        return _load().pkv_seq_len(self.handle)

    @property
    def num_blocks(self) -> int:
        return _load().pkv_seq_num_blocks(self.handle)

    def blocks(self) -> np.ndarray:
        lib = _load()
        return np.array([lib.pkv_seq_block(self.handle, j) for j in range(self.num_blocks)],
                        dtype=np.int32)

    def append(self, n: int):
        """Plan the append of n tokens: returns (slots int64[n], cow_pairs int64[k, 2])."""
        slots = np.empty(max(n, 1), dtype=np.int64)
        pair = np.empty(2, dtype=np.int64)
        cnt = ctypes.c_int32(0)
        rc = _load().pkv_seq_append_tokens(self.pool.handle, self.handle, n, slots.ctypes.data,
                                           pair.ctypes.data, ctypes.byref(cnt))
        if rc == -2:
            raise PoolExhausted("block pool exhausted")
        if rc != 0:
            raise ValueError(f"append rejected ({rc})")
        return slots[:n], pair.reshape(1, 2)[: cnt.value].copy()

    def fork(self) -> "Seq":
        h = _load().pkv_seq_fork(self.pool.handle, self.handle)
        if not h:
            raise MemoryError("fork failed")
        return Seq(self.pool, h)

    def release(self) -> None:
        if self.handle:
            _load().pkv_seq_release(self.pool.handle, self.handle)
            self.handle = 0


class BlockPool:
    """Free FIFO of block ids with refcounts (see include/pkv_pool.h)."""

    def __init__(self, num_blocks: int, block_size: int, seed: int = 0, shuffle: bool = True):
        self.handle = _load().pkv_pool_create(num_blocks, block_size, seed, int(shuffle))
        if not self.handle:
            raise ValueError("bad pool arguments")
        self.block_size = block_size

    def __del__(self):
        h = getattr(self, "handle", 0)
        if h and _lib is not None:
            _lib.pkv_pool_destroy(h)
            self.handle = 0

    @property
    def num_blocks(self) -> int:
        return _load().pkv_pool_num_blocks(self.handle)

    @property
    def num_free(self) -> int:
        return _load().pkv_pool_num_free(self.handle)

    def alloc(self) -> int:
        b = _load().pkv_pool_alloc(self.handle)
        if b < 0:
            raise PoolExhausted("block pool exhausted")
        return b

    def refcount(self, block: int) -> int:
        return _load().pkv_pool_refcount(self.handle, block)

    def incref(self, block: int) -> None:
        if _load().pkv_pool_incref(self.handle, block) != 0:
            raise ValueError(f"incref of unowned block {block}")

    def decref(self, block: int) -> None:
        if _load().pkv_pool_decref(self.handle, block) != 0:
            raise ValueError(f"decref of unowned block {block}")

    def new_seq(self) -> Seq:
        return Seq(self, _load().pkv_seq_create(self.handle))

    def block_tables(self, seqs, max_blocks: int | None = None):
        """Dense int32 [len(seqs), max_blocks] table padded with -1, and int32 lengths."""
        if max_blocks is None:
            max_blocks = max([s.num_blocks for s in seqs] + [1])
        n = len(seqs)
        handles = (ctypes.c_void_p * max(n, 1))(*[s.handle for s in seqs])
        tables = np.empty((n, max_blocks), dtype=np.int32)
        lens = np.empty(n, dtype=np.int32)
        rc = _load().pkv_build_block_tables(handles, n, max_blocks, tables.ctypes.data,
                                            lens.ctypes.data)
        if rc != 0:
            raise ValueError("a sequence has more blocks than max_blocks")
        return tables, lens
