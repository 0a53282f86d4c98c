"""CPU oracle for paged attention decode (fp64, plain C behind ctypes).

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the CPU
baseline leg of ``bench.py`` may import this package.  The product library
never loads it, and it shares no code with the CUDA path.

Every function follows "M5.3 - KV Memory Layout and Exact Reuse" (sections
named in ``pkv_oracle.h``), "7. Memory Management and Local Model State" and
the slot invariant of "Cache Concepts: Prefix Matching vs. Storage".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liboracle.so")

F32, BF16 = 0, 1
OK, BAD_ARG, BAD_SLOT, BAD_BLOCK = 0, 1, 2, 3
REJECT_VISIBILITY, REJECT_TABLE, REJECT_PHYSICAL = 10, 11, 12


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (-O2, OpenMP).  Returns the path."""
    src = os.path.join(_HERE, "pkv_oracle.c")
    hdr = os.path.join(_HERE, "pkv_oracle.h")
    if (not force and os.path.exists(LIB_PATH)
            and os.path.getmtime(LIB_PATH) >= max(os.path.getmtime(src), os.path.getmtime(hdr))):
        return LIB_PATH
    tmp = LIB_PATH + ".tmp"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
                           "-o", tmp, src, "-lm"])
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


_lib = None


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(LIB_PATH)
        i64, i32, vp, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_double
        p64 = ctypes.POINTER(ctypes.c_int64)
        lib.pkv_oracle_num_blocks.restype = i64
        lib.pkv_oracle_num_blocks.argtypes = [i64, i64]
        lib.pkv_oracle_tail_rows.restype = i64
        lib.pkv_oracle_tail_rows.argtypes = [i64, i64]
        lib.pkv_oracle_slot_id.restype = i64
        lib.pkv_oracle_slot_id.argtypes = [i64, i64, i64]
        lib.pkv_oracle_row_major_offset.restype = i64
        lib.pkv_oracle_row_major_offset.argtypes = [i32, vp, vp]
        lib.pkv_oracle_resolve.restype = i32
        lib.pkv_oracle_resolve.argtypes = [vp, i64, i64, i64, i64, i64, p64, p64]
        lib.pkv_oracle_slot_for_position.restype = i64
        lib.pkv_oracle_slot_for_position.argtypes = [vp, i64, i64]
        lib.pkv_oracle_slots_for_positions.restype = i32
        lib.pkv_oracle_slots_for_positions.argtypes = [vp, i64, vp, vp, i64, i64, vp]
        lib.pkv_oracle_kv_append.restype = i32
        lib.pkv_oracle_kv_append.argtypes = [i32, vp, vp, i64, i32, i32, i32, vp, vp, vp, i64]
        lib.pkv_oracle_kv_block_copy.restype = i32
        lib.pkv_oracle_kv_block_copy.argtypes = [i32, vp, vp, i64, i32, i32, i32, vp, i64]
        lib.pkv_oracle_paged_decode.restype = i32
        lib.pkv_oracle_paged_decode.argtypes = [i32, vp, vp, vp, i64, i32, i32, i32, vp, i32,
                                                vp, i32, i32, dbl, vp, vp, i32]
        lib.pkv_oracle_shared_prefix.restype = i32
        lib.pkv_oracle_shared_prefix.argtypes = [i32, vp, vp, vp, i64, i32, i32, i32, vp, i32,
                                                 vp, i32, vp, i32, i32, dbl, vp, vp, i32]
        lib.pkv_oracle_row_ledger.restype = i32
        lib.pkv_oracle_row_ledger.argtypes = [vp, i32, vp, i32, i64, i32, p64, p64]
        lib.pkv_oracle_expand_table.restype = i32
        lib.pkv_oracle_expand_table.argtypes = [vp, i64, i32, vp]
        lib.pkv_oracle_e4m3_decode.restype = dbl
        lib.pkv_oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.pkv_oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.pkv_oracle_e4m3_encode.argtypes = [dbl]
        lib.pkv_oracle_e4m3_encode_exhaustive.restype = ctypes.c_uint8
        lib.pkv_oracle_e4m3_encode_exhaustive.argtypes = [dbl]
        lib.pkv_oracle_mx_scale.restype = ctypes.c_uint8
        lib.pkv_oracle_mx_scale.argtypes = [dbl]
        lib.pkv_oracle_kv_append_mxfp8.restype = i32
        lib.pkv_oracle_kv_append_mxfp8.argtypes = [i32, vp, vp, i64, i32, i32, i32, vp, vp, vp, i64]
        lib.pkv_oracle_mxfp8_to_f32.restype = i32
        lib.pkv_oracle_mxfp8_to_f32.argtypes = [vp, i64, i32, i32, i32, vp]
        lib.pkv_oracle_chunk_tree.restype = i32
        lib.pkv_oracle_chunk_tree.argtypes = [i32, vp, vp, vp, i64, i32, i32, i32, vp, vp, vp, vp,
                                              i32, vp, i64, i32, i32, dbl, vp, vp, i32]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _dtype_code(a: np.ndarray) -> int:
    """float32 arrays are fp32 storage; uint16 arrays hold raw bf16 bits."""
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle storage must be float32 or uint16 (bf16 bits), got {a.dtype}")


# ---------------------------------------------------------------- index math
def num_blocks(num_tokens: int, block_size: int) -> int:
    return _load().pkv_oracle_num_blocks(num_tokens, block_size)


def tail_rows(num_tokens: int, block_size: int) -> int:
    return _load().pkv_oracle_tail_rows(num_tokens, block_size)


def slot_id(physical_slot: int, block_size: int, token_offset: int) -> int:
    return _load().pkv_oracle_slot_id(physical_slot, block_size, token_offset)


def row_major_offset(shape, coord) -> int:
    s = np.ascontiguousarray(shape, dtype=np.int64)
    c = np.ascontiguousarray(coord, dtype=np.int64)
    return _load().pkv_oracle_row_major_offset(len(s), _ptr(s), _ptr(c))


def resolve(table, context_len: int, block_size: int, num_pool_blocks: int, token: int):
    """Returns (status, physical_block, offset)."""
    t = np.ascontiguousarray(table, dtype=np.int32)
    blk, off = ctypes.c_int64(-1), ctypes.c_int64(-1)
    st = _load().pkv_oracle_resolve(_ptr(t), len(t), context_len, block_size,
                                    num_pool_blocks, token, ctypes.byref(blk), ctypes.byref(off))
    return st, blk.value, off.value


def slot_for_position(table, block_size: int, pos: int) -> int:
    t = np.ascontiguousarray(table, dtype=np.int32)
    return _load().pkv_oracle_slot_for_position(_ptr(t), block_size, pos)


def slots_for_positions(tables, block_size: int, rows, positions) -> np.ndarray:
    """slot_for_position for many (request, position) pairs: request rows[i]
    (a row of the 2-D int32 tables), position positions[i]."""
    t = np.ascontiguousarray(tables, dtype=np.int32)
    assert t.ndim == 2
    r = np.ascontiguousarray(rows, dtype=np.int32)
    p = np.ascontiguousarray(positions, dtype=np.int64)
    assert r.shape == p.shape
    out = np.empty(p.shape, np.int64)
    st = _load().pkv_oracle_slots_for_positions(_ptr(t), t.shape[1], _ptr(r), _ptr(p), p.size,
                                                block_size, _ptr(out))
    if st != OK:
        raise ValueError("slots_for_positions: a row, position or table bound is out of range")
    return out


# ---------------------------------------------------------------- data ops
def kv_append(k_cache: np.ndarray, v_cache: np.ndarray, k: np.ndarray, v: np.ndarray,
              slots: np.ndarray) -> int:
    """In place on k_cache/v_cache [NB, P, Hkv, D]; k, v: [N, Hkv, D]."""
    nb, p, hkv, d = k_cache.shape
    slots = np.ascontiguousarray(slots, dtype=np.int64)
    assert k.shape == (len(slots), hkv, d) and v.shape == k.shape
    assert k.dtype == k_cache.dtype == v.dtype == v_cache.dtype
    return _load().pkv_oracle_kv_append(_dtype_code(k_cache), _ptr(k_cache), _ptr(v_cache),
                                        nb, p, hkv, d, _ptr(np.ascontiguousarray(k)),
                                        _ptr(np.ascontiguousarray(v)), _ptr(slots), len(slots))


def kv_block_copy(k_cache: np.ndarray, v_cache: np.ndarray, pairs) -> int:
    nb, p, hkv, d = k_cache.shape
    pr = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
    return _load().pkv_oracle_kv_block_copy(_dtype_code(k_cache), _ptr(k_cache), _ptr(v_cache),
                                            nb, p, hkv, d, _ptr(pr), len(pr))


def paged_decode(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                 block_tables: np.ndarray, seq_lens: np.ndarray, scale: float,
                 nthreads: int = 1):
    """Returns (out [B, Hq, D] float64, lse [B, Hq] float64)."""
    nb, p, hkv, d = k_cache.shape
    b, hq, dq = q.shape
    assert dq == d and q.dtype == k_cache.dtype
    bt = np.ascontiguousarray(block_tables, dtype=np.int32).reshape(b, -1)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.zeros((b, hq, d), dtype=np.float64)
    lse = np.zeros((b, hq), dtype=np.float64)
    st = _load().pkv_oracle_paged_decode(_dtype_code(k_cache), _ptr(np.ascontiguousarray(q)),
                                         _ptr(k_cache), _ptr(v_cache), nb, p, hkv, d, _ptr(bt),
                                         bt.shape[1], _ptr(sl), b, hq, float(scale), _ptr(out),
                                         _ptr(lse), int(nthreads))
    if st != OK:
        raise ValueError(f"oracle paged_decode rejected its inputs (status {st})")
    return out, lse


def shared_prefix(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                  prefix_block_ids, prefix_len: int, suffix_block_tables: np.ndarray,
                  suffix_lens: np.ndarray, scale: float, nthreads: int = 1):
    nb, p, hkv, d = k_cache.shape
    b, hq, _ = q.shape
    pre = np.ascontiguousarray(prefix_block_ids, dtype=np.int32)
    st_ = np.ascontiguousarray(suffix_block_tables, dtype=np.int32).reshape(b, -1)
    sl = np.ascontiguousarray(suffix_lens, dtype=np.int32)
    out = np.zeros((b, hq, d), dtype=np.float64)
    lse = np.zeros((b, hq), dtype=np.float64)
    st = _load().pkv_oracle_shared_prefix(_dtype_code(k_cache), _ptr(np.ascontiguousarray(q)),
                                          _ptr(k_cache), _ptr(v_cache), nb, p, hkv, d, _ptr(pre),
                                          int(prefix_len), _ptr(st_), st_.shape[1], _ptr(sl), b, hq,
                                          float(scale), _ptr(out), _ptr(lse), int(nthreads))
    if st != OK:
        raise ValueError(f"oracle shared_prefix rejected its inputs (status {st})")
    return out, lse


def chunk_tree(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, chunks,
               block_ids, scale: float, nthreads: int = 1):
    """Attention over a prefix-tree snapshot by definition ([M5.3] 0x0BB,
    0x0BE): ``chunks`` is [n, 4] int rows (first id, rows, seq begin, seq
    end); each sequence attends to the concatenation of the chunks covering
    it.  Returns (out [B, Hq, D] float64, lse [B, Hq] float64)."""
    nb, p, hkv, d = k_cache.shape
    b, hq, dq = q.shape
    assert dq == d and q.dtype == k_cache.dtype
    ch = np.ascontiguousarray(chunks, dtype=np.int32).reshape(-1, 4)
    cols = [np.ascontiguousarray(ch[:, i]) for i in range(4)]
    ids = np.ascontiguousarray(block_ids, dtype=np.int32).reshape(-1)
    if ids.size == 0:
        ids = np.zeros(1, np.int32)
        n_ids = 0
    else:
        n_ids = ids.size
    out = np.zeros((b, hq, d), dtype=np.float64)
    lse = np.zeros((b, hq), dtype=np.float64)
    st = _load().pkv_oracle_chunk_tree(_dtype_code(k_cache), _ptr(np.ascontiguousarray(q)),
                                       _ptr(k_cache), _ptr(v_cache), nb, p, hkv, d,
                                       _ptr(cols[0]), _ptr(cols[1]), _ptr(cols[2]),
                                       _ptr(cols[3]), len(ch), _ptr(ids), n_ids, b, hq,
                                       float(scale), _ptr(out), _ptr(lse), int(nthreads))
    if st != OK:
        raise ValueError(f"oracle chunk_tree rejected its inputs (status {st})")
    return out, lse


# ------------------------------------------------------------------ MXFP8 pools
def e4m3_decode(code: int) -> float:
    """Value of an OCP FP8 E4M3 code."""
    return _load().pkv_oracle_e4m3_decode(int(code))


def e4m3_encode(x: float) -> int:
    """E4M3 code of x: nearest, ties to even, saturating at 448."""
    return int(_load().pkv_oracle_e4m3_encode(float(x)))


def e4m3_encode_exhaustive(x: float) -> int:
    """E4M3 code of x by searching every finite code for the nearest value."""
    return int(_load().pkv_oracle_e4m3_encode_exhaustive(float(x)))


def mx_scale(amax: float) -> int:
    """E8M0 scale byte of a 32-element group: smallest 2^(s - 127) with
    amax / 2^(s - 127) <= 448."""
    return int(_load().pkv_oracle_mx_scale(float(amax)))


def mxfp8_pool_bytes(num_blocks: int, block_size: int, num_kv_heads: int, head_dim: int) -> int:
    """Bytes of one MXFP8 cache buffer: the element plane, then the scale plane."""
    n = num_blocks * block_size * num_kv_heads * head_dim
    return n + n // 32


def kv_append_mxfp8(k_cache: np.ndarray, v_cache: np.ndarray, shape, k: np.ndarray,
                    v: np.ndarray, slot_mapping) -> int:
    """Quantize rows k, v ([N, Hkv, D], float32 or bf16 bits) into MXFP8
    pools (flat uint8 buffers of mxfp8_pool_bytes(*shape))."""
    nb, p, hkv, d = shape
    assert k_cache.dtype == np.uint8 and k_cache.size == mxfp8_pool_bytes(nb, p, hkv, d)
    sl = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    return _load().pkv_oracle_kv_append_mxfp8(_dtype_code(k), _ptr(k_cache), _ptr(v_cache), nb, p,
                                              hkv, d, _ptr(k), _ptr(v), _ptr(sl), len(sl))


def mxfp8_to_f32(cache: np.ndarray, shape) -> np.ndarray:
    """The fp32 values [NB, P, Hkv, D] an MXFP8 pool holds (exact)."""
    nb, p, hkv, d = shape
    out = np.empty((nb, p, hkv, d), np.float32)
    st = _load().pkv_oracle_mxfp8_to_f32(_ptr(cache), nb, p, hkv, d, _ptr(out))
    if st != OK:
        raise ValueError(f"oracle mxfp8_to_f32 rejected its inputs (status {st})")
    return out


def row_ledger(block_tables: np.ndarray, seq_lens: np.ndarray, num_pool_blocks: int,
               block_size: int):
    """Returns (logical_rows, unique_rows)."""
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32).reshape(len(sl), -1)
    lo, un = ctypes.c_int64(0), ctypes.c_int64(0)
    st = _load().pkv_oracle_row_ledger(_ptr(bt), bt.shape[1], _ptr(sl), len(sl),
                                       num_pool_blocks, block_size, ctypes.byref(lo),
                                       ctypes.byref(un))
    if st != OK:
        raise ValueError(f"oracle row_ledger rejected its inputs (status {st})")
    return lo.value, un.value


def expand_table(table, q: int) -> np.ndarray:
    """Kernel block ids for allocator block ids ([M5.3] 0x0AC): the last axis
    of ``table`` grows q-fold, allocator id a becoming a q .. a q + q - 1 and
    padding (-1) becoming q entries of -1."""
    t = np.ascontiguousarray(table, dtype=np.int32)
    out = np.empty(t.shape[:-1] + (t.shape[-1] * q,), np.int32)
    st = _load().pkv_oracle_expand_table(_ptr(t), t.size, q, _ptr(out))
    if st != OK:
        raise ValueError(f"oracle expand_table rejected its inputs (status {st})")
    return out
