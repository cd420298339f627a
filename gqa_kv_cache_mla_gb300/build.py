"""Build the kvw CUDA library (``libkvw.so``) in-tree for sm_103a.

Each ``csrc/*.cu`` file is compiled by nvcc in parallel
(``-gencode arch=compute_103a,code=sm_103a -O3 -lineinfo``) and linked into
one shared library with the CUDA runtime linked statically, so the library
only needs the NVIDIA driver at run time.  Objects go to ``_build/`` next to
this file.  Run ``python -m gqa_kv_cache_mla_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libkvw.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr", "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the kvw library needs the CUDA toolkit to build")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(INCLUDE, "kvw.h")]
    return any(os.path.getmtime(p) > t for p in deps)


def build_lib(csrc: str, out: str, objdir: str, verbose: bool = False, extra=()) -> str:
    """Compile every ``*.cu`` of ``csrc`` and link them into ``out``."""
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, "-I", csrc, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    srcs = sorted(glob.glob(os.path.join(csrc, "*.cu")))
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = out + ".tmp%d" % os.getpid()
    r = subprocess.run([cc, *ARCH, "-shared", "-cudart", "static", *objs, "-o", tmp],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, out)
    return out


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    """Build ``libkvw.so`` next to this file if any source is newer."""
    if not force and not _stale():
        return LIB
    return build_lib(CSRC, LIB, BUILD, verbose=verbose, extra=extra)


if __name__ == "__main__":
    v = "-v" in sys.argv
    print(build(force="--force" in sys.argv, verbose=v,
                extra=["-Xptxas", "-v"] if v else []))
