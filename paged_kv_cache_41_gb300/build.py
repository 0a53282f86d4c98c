"""Build the in-tree native libraries.

* ``libpkv.so``      -- the CUDA kernels and their C ABI (nvcc, sm_103a only).
* ``libpkv_pool.so`` -- the host block pool (gcc, plain C99).
* ``libpkv_probe.so`` -- read-only HBM streaming probes (bench.py's
  read-bandwidth denominator).
* ``tests/libpkv_wait_probe.so`` -- a test-only kernel for the bounded
  mbarrier wait (not part of libpkv).

The first three land next to this file.  Sources compile in parallel; nothing here uses
cmake or setuptools.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
CSRC = os.path.join(HERE, "csrc")

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

CUDA_SOURCES = [
    "pkv_api.cu",
    "kernels/append_copy.cu",
    "kernels/decode.cu",
    "kernels/decode_tc.cu",
    "kernels/decode_tc_mx.cu",
    "kernels/prefix_tc.cu",
    "kernels/tree.cu",
]
# Attention kernels take exp2/log2/division from the hardware approximations
# (softmax in base 2, well inside the attention tolerance).
PER_SOURCE_FLAGS = {
    "kernels/decode.cu": ["--use_fast_math"],
    "kernels/decode_tc.cu": ["--use_fast_math"],
    "kernels/decode_tc_mx.cu": ["--use_fast_math"],
    "kernels/prefix_tc.cu": ["--use_fast_math"],
    "kernels/tree.cu": ["--use_fast_math"],
}

LIB = os.path.join(HERE, "libpkv.so")
POOL_LIB = os.path.join(HERE, "libpkv_pool.so")


def _newer(target: str, deps) -> bool:
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(d) <= t for d in deps)


def _all_files(d, exts):
    out = []
    for root, _, files in os.walk(d):
        for f in files:
            if f.endswith(exts):
                out.append(os.path.join(root, f))
    return out


def build_pool(force=False) -> str:
    src = os.path.join(CSRC, "host", "pkv_pool.c")
    hdr = os.path.join(INCLUDE, "pkv_pool.h")
    if not force and _newer(POOL_LIB, [src, hdr]):
        return POOL_LIB
    tmp = POOL_LIB + ".tmp"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-I", INCLUDE,
                           "-o", tmp, src])
    os.replace(tmp, POOL_LIB)
    return POOL_LIB


def build_cuda(force=False, extra_flags=()) -> str:
    srcs = [os.path.join(CSRC, s) for s in CUDA_SOURCES if os.path.exists(os.path.join(CSRC, s))]
    deps = srcs + _all_files(CSRC, (".cuh", ".h")) + _all_files(INCLUDE, (".h",))
    if not force and not extra_flags and _newer(LIB, deps):
        return LIB
    objdir = os.path.join(ROOT, "_build")
    os.makedirs(objdir, exist_ok=True)
    common = [NVCC, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr", *extra_flags]
    procs, objs = [], []
    for s in srcs:
        obj = os.path.join(objdir, os.path.basename(s).replace(".cu", ".o"))
        objs.append(obj)
        extra = PER_SOURCE_FLAGS.get(os.path.relpath(s, CSRC), [])
        procs.append((s, subprocess.Popen(common + extra + ["-c", s, "-o", obj],
                                          stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for s, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append((s, out.decode(errors="replace")))
        elif out and os.environ.get("PKV_BUILD_VERBOSE"):
            sys.stderr.write(out.decode(errors="replace"))
    if failed:
        msg = "\n".join(f"--- {s}\n{o}" for s, o in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    tmp = LIB + ".tmp"
    subprocess.check_call([NVCC, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, LIB)
    return LIB


PROBE_SRC = os.path.join(CSRC, "probe", "hbm_read.cu")
PROBE_LIB = os.path.join(HERE, "libpkv_probe.so")


def build_probe(force=False) -> str:
    """The read-only HBM streaming probes that bench.py measures its
    read-bandwidth denominator with (csrc/probe/hbm_read.cu)."""
    deps = [PROBE_SRC, os.path.join(CSRC, "kernels", "common.cuh"), os.path.join(INCLUDE, "pkv.h")]
    if not force and _newer(PROBE_LIB, deps):
        return PROBE_LIB
    tmp = PROBE_LIB + ".tmp"
    subprocess.check_call([NVCC, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                           "-shared", "-I", INCLUDE, "-I", CSRC, "-o", tmp, PROBE_SRC])
    os.replace(tmp, PROBE_LIB)
    return PROBE_LIB


WAIT_PROBE_SRC = os.path.join(ROOT, "tests", "csrc", "wait_probe.cu")
WAIT_PROBE_LIB = os.path.join(ROOT, "tests", "libpkv_wait_probe.so")


def build_wait_probe(force=False) -> str:
    """The test suite's bounded-wait probe (tests/csrc/wait_probe.cu): its own
    small library over the kernels' common.cuh, not part of libpkv."""
    deps = [WAIT_PROBE_SRC, os.path.join(CSRC, "kernels", "common.cuh"),
            os.path.join(INCLUDE, "pkv.h")]
    if not force and _newer(WAIT_PROBE_LIB, deps):
        return WAIT_PROBE_LIB
    tmp = WAIT_PROBE_LIB + ".tmp"
    subprocess.check_call([NVCC, *ARCH, "-O2", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                           "-shared", "-I", INCLUDE, "-I", CSRC, "-o", tmp, WAIT_PROBE_SRC])
    os.replace(tmp, WAIT_PROBE_LIB)
    return WAIT_PROBE_LIB


def build_all(force=False) -> None:
    build_pool(force)
    build_cuda(force)
    build_probe(force)
    if os.path.exists(WAIT_PROBE_SRC):
        build_wait_probe(force)


if __name__ == "__main__":
    build_all(force="--force" in sys.argv)
