"""Build the in-tree shared library libsparse_mla.so for sm_103a with nvcc.

Each CUDA translation unit under csrc/ is compiled in parallel, then linked
into bwd_sparse_mla_gb300/libsparse_mla.so (the CUDA runtime is linked
statically; the library needs only the driver at run time).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libsparse_mla.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
          "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources() -> list:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _run(cmd: list) -> None:
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip() and os.environ.get("SMLA_BUILD_VERBOSE"):
        sys.stderr.write(r.stderr)


def build(extra_flags: list | None = None, lib: str = LIB, obj: str = OBJ) -> str:
    """Compile every translation unit and link `lib` (objects under `obj`).  The
    debug build (extra_flags=["-DSMLA_DEBUG"]) goes to its own paths, e.g.
    debug_paths(), so that it never replaces the product library."""
    os.makedirs(obj, exist_ok=True)
    cc = nvcc()
    flags = CFLAGS + list(extra_flags or [])
    srcs = sources()
    objs = [os.path.join(obj, os.path.basename(s)[:-3] + ".o") for s in srcs]
    with ThreadPoolExecutor(max_workers=max(1, len(srcs))) as ex:
        list(ex.map(lambda so: _run([cc, *ARCH, *flags, "-c", so[0], "-o", so[1]]), zip(srcs, objs)))
    tmp = lib + ".tmp"
    _run([cc, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, lib)
    return lib


def debug_paths() -> tuple:
    """(library, object folder) of the bounds-checked debug build."""
    d = os.path.join(PKG, "_build_debug")
    return os.path.join(d, "libsparse_mla_debug.so"), d


if __name__ == "__main__":
    flags = sys.argv[1:]
    # the bounds-checked debug build never replaces the product library
    print(build(flags, *debug_paths()) if "-DSMLA_DEBUG" in flags else build(flags))
