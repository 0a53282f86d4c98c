"""The C-ABI libraries load without a GPU and export every declared symbol."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "paged_kv_cache_41_gb300")


def _declared(header):
    text = open(os.path.join(ROOT, "include", header)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_\w+)\s*\(", text)))


def _exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib], capture_output=True, text=True,
                         check=True).stdout
    return {ln.split()[-1] for ln in out.splitlines() if ln.strip()}


@pytest.fixture(scope="module")
def libs():
    from paged_kv_cache_41_gb300 import build
    build.build_all()
    return os.path.join(PKG, "libpkv.so"), os.path.join(PKG, "libpkv_pool.so")


def test_pkv_header_symbols_exported(libs):
    lib, _ = libs
    names = _declared("pkv.h")
    assert "pkv_paged_attention_decode" in names and "pkv_kv_append" in names
    missing = set(names) - _exported(lib)
    assert not missing, missing
    ctypes.CDLL(lib)  # loads without a GPU


def test_pool_header_symbols_exported(libs):
    _, pool = libs
    names = _declared("pkv_pool.h")
    missing = set(names) - _exported(pool)
    assert not missing, missing


def test_binding_names_match_header(libs):
    from paged_kv_cache_41_gb300 import pkv
    assert set(pkv.EXPORTED) == set(_declared("pkv.h"))
    pkv.load_library()


def test_status_strings(libs):
    from paged_kv_cache_41_gb300 import pkv
    assert pkv.status_string(0) == "ok"
    assert "invalid" in pkv.status_string(1)
