"""Paged-KV attention decode for GB300 (sm_103a).

The device operations live in ``libpkv.so`` behind a C ABI (``include/pkv.h``);
:mod:`paged_kv_cache_41_gb300.pkv` is the thin ctypes binding with the same
names.  The host block pool (``include/pkv_pool.h``) is bound by
:mod:`paged_kv_cache_41_gb300.pool` and only generates inputs.
"""
__all__ = ["pkv", "pool", "workloads", "build"]
