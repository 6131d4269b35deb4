"""Builds the CUDA library ``libfa_attention.so`` in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into one shared
object next to this file.  A rebuild happens when a source or header is newer
than the library.  Usage: ``python -m exact_attention_37_gb300.build [-v] [-f] [--debug]``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libfa_attention.so")
OBJDIR = os.path.join(HERE, "_build")
# The debug build: the same sources with -DFA_DEBUG (device-side bounds, alignment
# and barrier-phase checks that record into the device error record, never trap).
LIB_DEBUG = os.path.join(HERE, "libfa_attention_debug.so")
OBJDIR_DEBUG = os.path.join(HERE, "_build_debug")
SOURCES = ["fa_api.cu", "fa_fwd.cu", "fa_bwd.cu", "fa_bwd_sq.cu", "fa_bwd256.cu", "fa_selftest.cu", "fa_host.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr", "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the attention library")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "fa_attention.h"))
    return files


def _flags_file(objdir: str) -> str:
    return os.path.join(objdir, "flags.txt")


def up_to_date(lib: str = LIB, objdir: str = OBJDIR, flags=()) -> bool:
    """The library exists, is newer than every source, and was built with `flags`."""
    if not os.path.exists(lib):
        return False
    try:
        with open(_flags_file(objdir)) as f:
            if f.read() != " ".join(flags):
                return False
    except OSError:
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(verbose: bool = False, force: bool = False, extra_flags=(), debug: bool = False,
          nvtx: bool | None = None) -> str:
    """Compile and link the library if needed; returns its path.  ``debug`` builds
    the checked variant (``libfa_attention_debug.so``) instead; ``nvtx`` (default:
    the FA_NVTX environment variable is set to 1) marks every C-ABI call with an
    NVTX range."""
    lib, objdir = (LIB_DEBUG, OBJDIR_DEBUG) if debug else (LIB, OBJDIR)
    if nvtx is None:
        nvtx = os.environ.get("FA_NVTX") == "1"
    extra_flags = (*extra_flags, *(["-DFA_DEBUG"] if debug else []), *(["-DFA_NVTX"] if nvtx else []))
    if not force and up_to_date(lib, objdir, extra_flags):
        return lib
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    errors = []
    for src, obj, r in results:
        if verbose and (r.stdout or r.stderr):
            print(f"--- {src}\n{r.stdout}{r.stderr}", file=sys.stderr)
        if r.returncode != 0:
            errors.append(f"{src}:\n{r.stderr}")
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    tmp = lib + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[obj for _, obj, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stderr)
    os.replace(tmp, lib)
    with open(_flags_file(objdir), "w") as f:
        f.write(" ".join(extra_flags))
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, debug="--debug" in sys.argv))
