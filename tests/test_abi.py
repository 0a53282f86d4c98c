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


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "pkv.h"
#include "pkv_pool.h"

/* A plain C caller of the ABI, without torch or the CUDA headers: host-side
 * validation and host-side planning need no GPU. */
int main(void) {
  pkv_cache_desc c;
  c.num_blocks = 8; c.block_size = 16; c.num_kv_heads = 2; c.head_dim = 64; c.dtype = PKV_BF16;
  if (strcmp(pkv_status_string(PKV_OK), "ok") != 0) return 10;
  /* null pools: rejected before any launch */
  if (pkv_kv_append(&c, NULL, NULL, NULL, NULL, NULL, 4, NULL) != PKV_ERR_INVALID_ARG) return 11;
  /* a bad descriptor */
  pkv_cache_desc bad = c;
  bad.head_dim = 96;
  if (pkv_kv_block_copy(&bad, NULL, NULL, NULL, 1, NULL) == PKV_OK) return 12;
  /* the prefix-tree planner runs on the host: one shared chunk, two leaves */
  pkv_chunk ch[3] = {{0, 20, 0, 2}, {2, 5, 0, 1}, {3, 7, 1, 2}};
  int32_t ids[4] = {0, 1, 2, 3};
  size_t pb = 0, wb = 0;
  pkv_status st = pkv_chunk_tree_plan(&c, ch, 3, ids, 4, 2, 8, -1, NULL, 0, &pb, &wb);
  if (st != PKV_OK || pb == 0) return 13;
  printf("c-abi ok %zu %zu\n", pb, wb);
  return 0;
}
"""


def test_plain_c_program_links_and_calls(libs, tmp_path):
    # include/pkv.h and pkv_pool.h compile as C99 on their own, and a C
    # program linked against libpkv.so calls it (host paths: no GPU needed)
    lib, _ = libs
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", PKG, "-lpkv", "-Wl,-rpath," + PKG],
                   check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, (out.returncode, out.stdout, out.stderr)
    assert out.stdout.startswith("c-abi ok")
