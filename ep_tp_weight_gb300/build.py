"""Build libumm.so (sm_103a) in-tree with nvcc: one object per translation
unit, compiled in parallel, linked with the static CUDA runtime."""
from __future__ import annotations

import glob
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(ROOT, "_build", "umm")
LIB = os.path.join(PKG, "libumm.so")
# the checked build: same sources with UMM_CHECKED (every copy-kernel access
# tested against its buffer's bounds and alignment), for tests
CHECKED_OBJDIR = os.path.join(ROOT, "_build", "umm_checked")
CHECKED_LIB = os.path.join(PKG, "libumm_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None,
          checked: bool = False) -> str:
    """Compile libumm.so (or, with checked=True, libumm_checked.so) in-tree."""
    lib, objdir = (CHECKED_LIB, CHECKED_OBJDIR) if checked else (LIB, OBJDIR)
    if not force and not stale(lib):
        return lib
    os.makedirs(objdir, exist_ok=True)
    extra = list(extra or []) + (["-DUMM_CHECKED"] if checked else [])

    def compile_one(src: str) -> str:
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        cmd = ["nvcc", *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd))
        subprocess.check_call(cmd)
        return obj

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = lib + f".tmp{os.getpid()}"
    subprocess.check_call(["nvcc", *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, lib)
    return lib


CEILING_SRC = os.path.join(CSRC, "ceiling", "mix_ceiling.cu")
CEILING_EXE = os.path.join(ROOT, "_build", "mix_ceiling")


def build_ceiling(force: bool = False) -> str:
    """Compile the read:write-mix ceiling program (a standalone executable,
    not part of libumm) for `bench.py --ceilings`."""
    if force or not os.path.exists(CEILING_EXE) or os.path.getmtime(CEILING_SRC) > os.path.getmtime(CEILING_EXE):
        os.makedirs(os.path.dirname(CEILING_EXE), exist_ok=True)
        tmp = CEILING_EXE + f".tmp{os.getpid()}"
        subprocess.check_call(["nvcc", *ARCH, "-O3", "-std=c++17", "-o", tmp, CEILING_SRC])
        os.replace(tmp, CEILING_EXE)
    return CEILING_EXE


def build_all(force: bool = False) -> None:
    """Both libraries, compiled side by side."""
    with ThreadPoolExecutor(max_workers=2) as ex:
        list(ex.map(lambda c: build(force=force, checked=c), (False, True)))


if __name__ == "__main__":
    build(force=True, verbose=True)
    build(force=True, verbose=True, checked=True)
