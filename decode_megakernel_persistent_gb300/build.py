"""Build libll.so (the C-ABI library) in-tree with nvcc for sm_103a.

Five translation units are compiled in parallel and linked into
``decode_megakernel_persistent_gb300/libll.so`` with the CUDA runtime linked
statically, so the library needs nothing but the driver at run time.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libll.so")
SOURCES = ("mk_cuda_cores.cu", "mk_tensor_cores.cu", "mk_geo.cu", "chain.cu", "schedule.cpp", "api.cpp",
           "static_step.cu", "prefill.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(ROOT, "include", "ll.h"))
    return files


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    if os.environ.get("LL_DEBUG_CHECKS") == "1" or os.environ.get("LL_RING"):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-I", os.path.join(ROOT, "include")]
    if verbose:
        flags += ["-Xptxas", "-v"]
    if os.environ.get("LL_DEBUG_CHECKS") == "1":
        # self-checking build: every hot-path index is bounds-checked on the device
        flags += ["-DLL_DEBUG_CHECKS"]
    ring = os.environ.get("LL_RING")
    if ring:
        # another shared-memory ring geometry, for comparisons: "<pages>x<KB>", the
        # 192 KB total kept (12x16 also cuts batches to 2 sequences for room)
        pages, kb = (int(v) for v in ring.lower().split("x"))
        flags += [f"-DLL_NPAGES={pages}", f"-DLL_PAGE_BYTES={kb * 1024}"]
        if pages * kb != 192:
            raise ValueError("LL_RING must keep 192 KB of pages")
        if pages > 8:
            flags += ["-DLL_MAX_B=2"]

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            print(log)
    tmp = LIB + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
