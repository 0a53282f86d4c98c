"""Thin Python binding of libpkv (``include/pkv.h``) with the same names.

Argument marshalling only: torch tensors supply device memory and the current
CUDA stream; every step of the computation runs in the library's kernels.
There is no fallback: if ``libpkv.so`` is missing or a call is rejected, the
binding raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA, PKV_ERR_DEVICE, PKV_ERR_CAPACITY = range(6)
# PKV_STATIC_SCRATCH_BYTES of include/pkv.h: the library-owned scratch array
STATIC_SCRATCH_BYTES = 16 << 20
PKV_F32, PKV_BF16, PKV_MXFP8 = 0, 1, 2
DEVERR_SLOT, DEVERR_BLOCK, DEVERR_LENGTH, DEVERR_TIMEOUT = 1, 2, 4, 8

EXPORTED = [
    "pkv_kv_append",
    "pkv_kv_block_copy",
    "pkv_decode_workspace_bytes",
    "pkv_decode_num_ctas",
    "pkv_expand_block_tables",
    "pkv_paged_attention_decode",
    "pkv_paged_attention_decode_static",
    "pkv_shared_prefix_workspace_bytes",
    "pkv_shared_prefix_attention",
    "pkv_prefix_split_len",
    "pkv_prefix_attention_states",
    "pkv_chunk_tree_plan",
    "pkv_chunk_tree_attention",
    "pkv_get_device_error",
    "pkv_status_string",
]


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int64), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


_lib = None


def load_library():
    """Load libpkv.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing; build it with paged_kv_cache_41_gb300.build")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
    dp = ctypes.POINTER(CacheDesc)
    lib.pkv_kv_append.restype = ctypes.c_int
    lib.pkv_kv_append.argtypes = [dp, vp, vp, vp, vp, vp, i64, vp]
    lib.pkv_kv_block_copy.restype = ctypes.c_int
    lib.pkv_kv_block_copy.argtypes = [dp, vp, vp, vp, i64, vp]
    lib.pkv_decode_workspace_bytes.restype = ctypes.c_size_t
    lib.pkv_decode_workspace_bytes.argtypes = [dp, i32, i32, i32, i32]
    lib.pkv_expand_block_tables.restype = i32
    lib.pkv_expand_block_tables.argtypes = [vp, i32, i32, i32, i32, vp, vp]
    lib.pkv_decode_num_ctas.restype = i32
    lib.pkv_decode_num_ctas.argtypes = [dp, i32, i32, i32, i32]
    lib.pkv_paged_attention_decode.restype = ctypes.c_int
    lib.pkv_paged_attention_decode.argtypes = [dp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, f32,
                                               i32, vp, ctypes.c_size_t, vp]
    lib.pkv_paged_attention_decode_static.restype = ctypes.c_int
    lib.pkv_paged_attention_decode_static.argtypes = [dp, vp, vp, vp, vp, vp, vp, i32, vp, i32,
                                                      i32, f32, i32, vp]
    lib.pkv_shared_prefix_workspace_bytes.restype = ctypes.c_size_t
    lib.pkv_shared_prefix_workspace_bytes.argtypes = [dp, i32, i32, i32, i32, i32]
    lib.pkv_shared_prefix_attention.restype = ctypes.c_int
    lib.pkv_shared_prefix_attention.argtypes = [dp, vp, vp, vp, vp, vp, vp, i32, vp, i32, vp, i32,
                                                i32, f32, i32, vp, ctypes.c_size_t, vp]
    lib.pkv_prefix_split_len.restype = i32
    lib.pkv_prefix_split_len.argtypes = [dp, i32, i32, i32]
    lib.pkv_prefix_attention_states.restype = ctypes.c_int
    lib.pkv_prefix_attention_states.argtypes = [dp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32,
                                                vp]
    lib.pkv_chunk_tree_plan.restype = ctypes.c_int
    lib.pkv_chunk_tree_plan.argtypes = [dp, vp, i32, vp, i64, i32, i32, i32, vp, ctypes.c_size_t,
                                        ctypes.POINTER(ctypes.c_size_t),
                                        ctypes.POINTER(ctypes.c_size_t)]
    lib.pkv_chunk_tree_attention.restype = ctypes.c_int
    lib.pkv_chunk_tree_attention.argtypes = [dp, vp, vp, vp, vp, vp, i32, i32, f32, vp, vp, vp,
                                             ctypes.c_size_t, vp]
    lib.pkv_get_device_error.restype = ctypes.c_int
    lib.pkv_get_device_error.argtypes = [ctypes.POINTER(i32), vp]
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_status_string.argtypes = [ctypes.c_int]
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().pkv_status_string(status).decode()


def _check(status: int, what: str):
    if status != PKV_OK:
        raise PkvError(status, what)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


class MxPool:
    """An MXFP8 K (or V) pool (include/pkv.h): one uint8 device buffer holding
    the E4M3 element plane [num_blocks, block_size, num_kv_heads, head_dim]
    followed by the E8M0 scale plane [num_blocks, num_kv_heads, block_size,
    head_dim / 32].  q, k, v and out beside it are bf16."""

    def __init__(self, num_blocks, block_size, num_kv_heads, head_dim, device="cuda", fill=0):
        self.shape = (int(num_blocks), int(block_size), int(num_kv_heads), int(head_dim))
        n = num_blocks * block_size * num_kv_heads * head_dim
        self.plane_bytes = n
        self.buf = torch.full((n + n // 32,), fill, dtype=torch.uint8, device=device)

    @property
    def device(self):
        return self.buf.device

    def data_ptr(self) -> int:
        return self.buf.data_ptr()

    @property
    def elements(self) -> torch.Tensor:
        """The element plane as raw E4M3 codes (uint8)."""
        return self.buf[:self.plane_bytes].view(self.shape)

    @property
    def scales(self) -> torch.Tensor:
        """The scale plane (E8M0 bytes)."""
        nb, p, hkv, d = self.shape
        return self.buf[self.plane_bytes:].view(nb, hkv, p, d // 32)


def cache_desc(k_cache) -> CacheDesc:
    """Descriptor of a [num_blocks, block_size, num_kv_heads, head_dim] pool
    (a bf16 or fp32 tensor, or an MxPool)."""
    if isinstance(k_cache, MxPool):
        nb, p, hkv, d = k_cache.shape
        return CacheDesc(nb, p, hkv, d, PKV_MXFP8)
    if k_cache.dim() != 4 or not k_cache.is_contiguous():
        raise ValueError("cache must be a contiguous [NB, P, Hkv, D] tensor")
    if k_cache.dtype == torch.bfloat16:
        dt = PKV_BF16
    elif k_cache.dtype == torch.float32:
        dt = PKV_F32
    else:
        raise TypeError(f"unsupported cache dtype {k_cache.dtype}")
    nb, p, hkv, d = k_cache.shape
    return CacheDesc(nb, p, hkv, d, dt)


def kv_append(k_cache, v_cache, k, v, slot_mapping, stream=None) -> None:
    """Scatter rows k[i], v[i] ([N, Hkv, D]) into slot slot_mapping[i] (int64)."""
    desc = cache_desc(k_cache)
    _check(load_library().pkv_kv_append(ctypes.byref(desc), _ptr(k_cache), _ptr(v_cache),
                                        _ptr(k.contiguous()), _ptr(v.contiguous()),
                                        _ptr(slot_mapping), slot_mapping.numel(), _stream(stream)),
           "pkv_kv_append")


def kv_block_copy(k_cache, v_cache, src_dst_pairs, stream=None) -> None:
    """Copy whole blocks src -> dst for each row of int64 [n, 2] pairs."""
    desc = cache_desc(k_cache)
    n = src_dst_pairs.shape[0] if src_dst_pairs.numel() else 0
    _check(load_library().pkv_kv_block_copy(ctypes.byref(desc), _ptr(k_cache), _ptr(v_cache),
                                            _ptr(src_dst_pairs), n, _stream(stream)),
           "pkv_kv_block_copy")


def decode_workspace_bytes(k_cache, num_seqs, num_q_heads, max_blocks_per_seq,
                           partition_size=0) -> int:
    desc = cache_desc(k_cache)
    return load_library().pkv_decode_workspace_bytes(ctypes.byref(desc), num_seqs, num_q_heads,
                                                     max_blocks_per_seq, partition_size)


def expand_block_tables(tables, alloc_block_size, kernel_block_size, out=None, stream=None):
    """Kernel-visible tables for a pool of P_a-row allocator blocks read as
    P_k-row kernel blocks (include/pkv.h): int32 [B, max_blocks * P_a / P_k]."""
    b, m = tables.shape
    q = alloc_block_size // kernel_block_size if kernel_block_size > 0 else 0
    if out is None:
        out = torch.empty(b, m * max(q, 1), dtype=torch.int32, device=tables.device)
    _check(load_library().pkv_expand_block_tables(_ptr(tables), b, m, alloc_block_size,
                                                  kernel_block_size, _ptr(out), _stream(stream)),
           "pkv_expand_block_tables")
    return out


def decode_num_ctas(k_cache, num_seqs, num_q_heads, max_blocks_per_seq, partition_size=0) -> int:
    desc = cache_desc(k_cache)
    return load_library().pkv_decode_num_ctas(ctypes.byref(desc), num_seqs, num_q_heads,
                                              max_blocks_per_seq, partition_size)


def paged_attention_decode(q, k_cache, v_cache, block_tables, seq_lens, scale, *, out=None,
                           lse=None, partition_size=0, workspace=None, stream=None):
    """Attention of q [B, Hq, D] over each sequence's paged history.

    block_tables: int32 [B, max_blocks]; seq_lens: int32 [B].  Returns out
    (and writes lse [B, Hq] float32 when given).  The workspace is allocated
    here through torch when not supplied.
    """
    desc = cache_desc(k_cache)
    b, hq, _ = q.shape
    max_blocks = block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    need = load_library().pkv_decode_workspace_bytes(ctypes.byref(desc), b, hq, max_blocks,
                                                     partition_size) if b else 0
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load_library().pkv_paged_attention_decode(
        ctypes.byref(desc), _ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_tables), max_blocks, _ptr(seq_lens), b, hq, float(scale), partition_size,
        _ptr(workspace), ws_bytes, _stream(stream)), "pkv_paged_attention_decode")
    return out


def paged_attention_decode_static(q, k_cache, v_cache, block_tables, seq_lens, scale, *,
                                  out=None, lse=None, partition_size=0, stream=None):
    """Allocation-free paged decode: the decode's workspace is the library's
    own fixed device array (include/pkv.h), so no workspace is
    passed and nothing is allocated by the call itself.  For callers that may
    not allocate device memory.  Raises PkvError (status PKV_ERR_CAPACITY) when
    the sizes need more than STATIC_SCRATCH_BYTES of scratch.  Calls that could
    overlap on the GPU share that array and must be ordered."""
    desc = cache_desc(k_cache)
    b, hq, _ = q.shape
    if out is None:
        out = torch.empty_like(q)
    _check(load_library().pkv_paged_attention_decode_static(
        ctypes.byref(desc), _ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), b, hq, float(scale),
        partition_size, _stream(stream)), "pkv_paged_attention_decode_static")
    return out


def shared_prefix_workspace_bytes(k_cache, num_seqs, num_q_heads, prefix_len,
                                  max_suffix_blocks, partition_size=0) -> int:
    desc = cache_desc(k_cache)
    return load_library().pkv_shared_prefix_workspace_bytes(
        ctypes.byref(desc), num_seqs, num_q_heads, prefix_len, max_suffix_blocks, partition_size)


def shared_prefix_attention(q, k_cache, v_cache, prefix_block_ids, prefix_len,
                            suffix_block_tables, suffix_lens, scale, *, out=None, lse=None,
                            partition_size=0, workspace=None, stream=None):
    """Attention over prefix ++ suffix for every request, with the shared
    prefix as one tensor-core contraction per kv head (include/pkv.h)."""
    desc = cache_desc(k_cache)
    b, hq, _ = q.shape
    max_suffix = suffix_block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    need = shared_prefix_workspace_bytes(k_cache, b, hq, prefix_len, max_suffix,
                                         partition_size) if b else 0
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load_library().pkv_shared_prefix_attention(
        ctypes.byref(desc), _ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache),
        _ptr(prefix_block_ids), int(prefix_len), _ptr(suffix_block_tables), max_suffix,
        _ptr(suffix_lens), b, hq, float(scale), partition_size, _ptr(workspace), ws_bytes,
        _stream(stream)), "pkv_shared_prefix_attention")
    return out


def prefix_split_len(k_cache, num_seqs, num_q_heads, prefix_len) -> int:
    desc = cache_desc(k_cache)
    return load_library().pkv_prefix_split_len(ctypes.byref(desc), num_seqs, num_q_heads,
                                               prefix_len)


def prefix_attention_states(q, k_cache, v_cache, prefix_block_ids, prefix_len, scale, *,
                            split_len=0, states_o=None, states_lse=None, stream=None):
    """Per-split (O, LSE) states of every query row against the shared prefix
    (include/pkv.h).  Returns (states_o [B, Hq, n, D] fp32, states_lse
    [B, Hq, n] fp32 natural log, split_len)."""
    desc = cache_desc(k_cache)
    b, hq, d = q.shape
    if split_len == 0:
        split_len = prefix_split_len(k_cache, b, hq, prefix_len)
    n = (prefix_len + split_len - 1) // split_len if split_len else 0
    if states_o is None:
        states_o = torch.empty(b, hq, n, d, dtype=torch.float32, device=q.device)
    if states_lse is None:
        states_lse = torch.empty(b, hq, n, dtype=torch.float32, device=q.device)
    _check(load_library().pkv_prefix_attention_states(
        ctypes.byref(desc), _ptr(states_o), _ptr(states_lse), _ptr(q), _ptr(k_cache),
        _ptr(v_cache), _ptr(prefix_block_ids), int(prefix_len), int(split_len), b, hq, float(scale),
        _stream(stream)), "pkv_prefix_attention_states")
    return states_o, states_lse, split_len


class ChunkTreePlan:
    """A planned prefix-tree snapshot (include/pkv.h): the plan's host bytes,
    their device copy, and the workspace the attention needs."""

    def __init__(self, host, device, workspace_bytes, num_seqs, num_q_heads):
        self.host = host
        self.device = device
        self.workspace_bytes = workspace_bytes
        self.num_seqs = num_seqs
        self.num_q_heads = num_q_heads


def chunk_tree_plan(k_cache, chunks, block_ids, num_seqs, num_q_heads, threshold=-1,
                    device=None, host_buffer=None, device_buffer=None) -> ChunkTreePlan:
    """Plan a tree snapshot.  ``chunks``: int [n, 4] rows (first id, rows,
    seq begin, seq end) in tree order; ``block_ids``: int32 block ids; both
    host data.  The plan's bytes are copied to ``device`` (default: the
    cache's device) with torch.  A serving loop that re-plans every step can
    pass uint8 buffers to reuse: ``host_buffer`` (pinned, so the copy is
    asynchronous: do not re-plan into it before that copy has run) and
    ``device_buffer``."""
    desc = cache_desc(k_cache)
    ch = np.ascontiguousarray(np.asarray(chunks, dtype=np.int32).reshape(-1, 4))
    ids = np.ascontiguousarray(np.asarray(block_ids, dtype=np.int32).reshape(-1))
    lib = load_library()
    pb, wb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    args = (ctypes.byref(desc), ctypes.c_void_p(ch.ctypes.data), len(ch),
            ctypes.c_void_p(ids.ctypes.data), ids.size, int(num_seqs), int(num_q_heads),
            int(threshold))
    _check(lib.pkv_chunk_tree_plan(*args, None, 0, ctypes.byref(pb), ctypes.byref(wb)),
           "pkv_chunk_tree_plan")
    n = pb.value
    if host_buffer is not None and host_buffer.numel() >= n:
        host = host_buffer[:n]
    else:
        host = torch.zeros(n, dtype=torch.uint8)
    _check(lib.pkv_chunk_tree_plan(*args, _ptr(host), n, ctypes.byref(pb), ctypes.byref(wb)),
           "pkv_chunk_tree_plan")
    if device_buffer is not None and device_buffer.numel() >= n:
        dev = device_buffer[:n]
        dev.copy_(host, non_blocking=host.is_pinned())
    else:
        dev = host.to(device if device is not None else k_cache.device)
    return ChunkTreePlan(host, dev, wb.value, int(num_seqs), int(num_q_heads))


def chunk_tree_attention(q, k_cache, v_cache, plan: ChunkTreePlan, scale, *, out=None, lse=None,
                         workspace=None, stream=None):
    """Attention of every sequence over its path of the planned tree
    (include/pkv.h).  Returns out [B, Hq, D]."""
    desc = cache_desc(k_cache)
    b, hq, _ = q.shape
    if out is None:
        out = torch.empty_like(q)
    if workspace is None and plan.workspace_bytes:
        workspace = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load_library().pkv_chunk_tree_attention(
        ctypes.byref(desc), _ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), b, hq,
        float(scale), _ptr(plan.host), _ptr(plan.device), _ptr(workspace), ws_bytes,
        _stream(stream)), "pkv_chunk_tree_attention")
    return out


def get_device_error(stream=None) -> int:
    """Synchronise, read and clear the device error word (PKV_DEVERR_* bits)."""
    code = ctypes.c_int32(0)
    st = load_library().pkv_get_device_error(ctypes.byref(code), _stream(stream))
    if st not in (PKV_OK, PKV_ERR_DEVICE):
        raise PkvError(st, "pkv_get_device_error")
    return code.value
