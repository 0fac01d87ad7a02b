"""Build the CUDA library ``libpa_gb300.so`` in-tree (sm_103a only).

Each ``csrc/*.cu`` compiles to an object in parallel with nvcc, then one link
step makes the shared library next to this file. The CUDA runtime is linked
statically and the driver is reached at run time through the runtime's
entry-point query, so the library loads (and its exports can be listed) on a
machine without a GPU driver.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpa_gb300.so")
# Test build: the same sources with PA_PDUMP defined, which makes the FP8
# kernels write every probability code they hand to the P V MMA to a buffer
# the tests provide (include/attn_pdump.h). Never the library that is timed.
PDUMP_OBJ = os.path.join(HERE, "_build_pdump")
PDUMP_LIB = os.path.join(HERE, "libpa_gb300_pdump.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I", INCLUDE, "-I", SRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources() -> list[str]:
    return sorted(os.path.join(SRC, f) for f in os.listdir(SRC) if f.endswith(".cu"))


def _deps() -> list[str]:
    files = sources() + [os.path.join(SRC, f) for f in os.listdir(SRC) if f.endswith((".h", ".cuh"))]
    return files + [os.path.join(INCLUDE, "attn.h"), os.path.join(INCLUDE, "attn_pdump.h")]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          pdump: bool = False) -> str:
    """Build libpa_gb300.so (or, with pdump=True, the test build libpa_gb300_pdump.so)."""
    lib, objdir = (PDUMP_LIB, PDUMP_OBJ) if pdump else (LIB, OBJ)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(objdir, exist_ok=True)
    exe = nvcc()
    flags = NVCC_FLAGS + list(extra_flags or []) + (["-DPA_PDUMP"] if pdump else [])

    def compile_one(src: str) -> str:
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        cmd = [exe, *ARCH, *flags, "-c", src, "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        if verbose and (res.stdout or res.stderr):
            print(res.stdout + res.stderr, file=sys.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + f".{os.getpid()}.tmp"
    cmd = [exe, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    v = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None
    print(build(force=True, verbose=v or bool(extra), extra_flags=extra))
