"""Builds liblayoutcopy.so (the C-ABI library) in-tree for sm_103a.

The translation units are compiled in parallel with nvcc and linked into one
shared object next to this file; the CUDA runtime is linked statically and
the driver is reached through the runtime's entry-point query, so the library
needs nothing but libcuda at run time.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_NAME = "liblayoutcopy.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)

SOURCES = ["plan.cpp", "api.cu", "host_copy.cu", "host_copy_static.cu", "k_vec.cu", "k_warp.cu", "k_shuffle.cu", "k_staged.cu",
           "k_warp_w1.cu", "k_warp_w2.cu", "k_warp_w4.cu", "k_warp_w8.cu", "k_warp_w16.cu",
           "k_tile.cu", "k_smem.cu", "k_tma_copy.cu", "k_stencil.cu", "k_loop.cu"]
HEADERS = ["lc_internal.h", "ptx.cuh", "device_common.cuh", "launch.h", "k_warp.cuh", "tensor_map.h", "bulk_store.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O3",
          "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC)")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files += [os.path.join(INCLUDE, h) for h in ("layout_copy.h", "layout_copy_device.cuh")]
    files.append(os.path.abspath(__file__))
    return files


def _stale(target: str) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          out: str | None = None, defines=(), only=None) -> str:
    """Compile and link if any input changed; returns the library path.

    ``out`` / ``defines`` build a variant (compile-time knobs such as
    LC_TILE_ROWS_W1) into another file; the in-tree library is the default
    build.  ``only`` (a variant build) compiles just those sources with the
    defines and links them with the default build's other objects.
    """
    lib_path = out or LIB_PATH
    build_dir = BUILD_DIR if out is None else out + ".objs"
    if not force and not _stale(lib_path):
        return lib_path
    if only is not None and out is not None:
        build()  # the default objects the variant links with
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    extra = ["-D" + d for d in defines]

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, "-c", os.path.join(CSRC, src), "-o", obj] + ARCH + COMMON + extra
        if ptxas_info and src.endswith(".cu"):
            cmd += ["-Xptxas", "-v"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), res.stderr))
        if verbose or ptxas_info:
            sys.stderr.write(res.stderr)
        return obj

    todo = SOURCES if only is None or out is None else [x for x in SOURCES if x in only]
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        built = dict(zip(todo, ex.map(compile_one, todo)))
    objs = [built.get(x) or os.path.join(BUILD_DIR, os.path.splitext(x)[0] + ".o") for x in SOURCES]
    tmp = lib_path + ".%d.tmp" % os.getpid()
    cmd = [cc, "-shared", "-o", tmp] + objs + ARCH + ["-Xcompiler", "-fPIC"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), res.stderr))
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
