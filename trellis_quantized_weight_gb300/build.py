"""Builds libtrellis_gb300.so in-tree with nvcc for sm_103a.

One object per translation unit under csrc/, compiled in parallel, then linked
into ``_build/libtrellis_gb300.so`` next to this file.  No cmake, no torch
extension machinery: the library is a plain C-ABI shared object.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB_NAME = "libtrellis_gb300.so"
LIB_PATH = os.path.join(BUILD, LIB_NAME)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# Host code with hidden visibility: the library exports only the C ABI (marked
# in include/trellis.h), so its internal statics stay private to each copy.
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2,-fvisibility=hidden",
              "--expt-relaxed-constexpr"]


def cuda_home() -> str:
    for cand in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return cand
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    raise RuntimeError("nvcc not found: set CUDA_HOME")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers() -> list[str]:
    return (glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, jobs: int | None = None,
          defines: tuple[str, ...] = (), build_dir: str | None = None) -> str:
    """Compile and link the library if any source or header is newer than it.

    ``defines`` (nvcc -D) with a separate ``build_dir`` make another copy of the
    library, e.g. the trace build (``TRELLIS_TRACE``, see trace.py); the shipped
    library is the one built with neither."""
    home = cuda_home()
    nvcc = os.path.join(home, "bin", "nvcc")
    out_dir = build_dir or BUILD
    lib_path = os.path.join(out_dir, LIB_NAME)
    flags = [*NVCC_FLAGS, *(f"-D{d}" for d in defines)]
    os.makedirs(os.path.join(out_dir, "obj"), exist_ok=True)
    srcs = sources()
    headers = _headers()
    objs = [os.path.join(out_dir, "obj", os.path.basename(s)[:-3] + ".o") for s in srcs]

    def compile_one(src_obj):
        src, obj = src_obj
        if not force and not _stale(obj, [src] + headers):
            return None
        cmd = [nvcc, *ARCH, *flags, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj + ".tmp"]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        os.replace(obj + ".tmp", obj)
        return r.stderr if verbose else None

    jobs = jobs or min(len(srcs), os.cpu_count() or 4)
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        for out in ex.map(compile_one, zip(srcs, objs)):
            if out:
                print(out)

    if force or _stale(lib_path, objs):
        libdir = os.path.join(home, "lib64")
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", lib_path + ".tmp", *objs,
               "-Xlinker", f"-rpath,{libdir}"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(lib_path + ".tmp", lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
