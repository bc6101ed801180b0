"""Build libkvq.so in-tree with nvcc for sm_103a (GB300).

Each CUDA translation unit compiles in its own nvcc process (in parallel),
then one link step makes the shared library next to this file.  Up-to-date
objects are reused.  build(debug=True) makes libkvq_debug.so, the same
sources with -DKVQ_BOUNDS_CHECK (device-side bounds checks that report
KVQ_DEVERR_BOUNDS), in its own object folder.  Run as ``python sub_byte_quantized_write_gb300/build_lib.py`` (the
package itself cannot be imported before the library exists).
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libkvq.so")
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "libkvq_debug.so")
SOURCES = ["kvq_api.cu", "kvq_write.cu", "kvq_decode.cu", "kvq_prefill_tc.cu"]
HEADERS = ["kvq_common.cuh", "kvq_internal.h", "kvq_tc.cuh", "kvq_row.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _newest_dep() -> float:
    deps = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "kvq.h"), __file__]
    return max(os.path.getmtime(p) for p in deps)


def _compile(src: str, extra, build_dir: str) -> str:
    obj = os.path.join(build_dir, src.replace(".cu", ".o"))
    path = os.path.join(CSRC, src)
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(path), _newest_dep()):
        return obj
    cmd = [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
           "-diag-suppress", "177", "-c", path, "-o", obj + ".tmp", *extra]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    os.replace(obj + ".tmp", obj)
    return obj


def build(verbose_ptxas: bool = False, debug: bool = False) -> str:
    build_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    os.makedirs(build_dir, exist_ok=True)
    extra = (["-Xptxas", "-v"] if verbose_ptxas else []) + (["-DKVQ_BOUNDS_CHECK"] if debug else [])
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, build_dir), SOURCES))
    if os.path.exists(lib) and os.path.getmtime(lib) >= max(os.path.getmtime(o) for o in objs):
        return lib
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose_ptxas="-v" in sys.argv, debug="--debug" in sys.argv))
