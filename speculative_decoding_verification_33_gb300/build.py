"""In-tree build of the verify library (``_build/libspecverify.so``) for sm_103a with nvcc.

The translation units are compiled in parallel and linked into one shared library with the
CUDA runtime linked statically. No CMake, no torch extension machinery.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libspecverify.so"
SOURCES = ["sv_kernel.cu", "sv_api.cu", "sv_probe.cu", "sv_rows.cu", "sv_lmhead.cu",
           "sv_hverify.cu", "sv_greedy.cu", "sv_small.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
         "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the verify library needs the CUDA 13 toolkit")
    return exe


def lib_path() -> str:
    return os.path.join(OUT_DIR, LIB_NAME)


def source_digest() -> str:
    """Hash of every source and header the library is built from."""
    h = hashlib.sha256()
    files = sorted(os.listdir(CSRC)) + ["../../include/" + f for f in sorted(os.listdir(INCLUDE))]
    for f in files:
        p = os.path.normpath(os.path.join(CSRC, f))
        if os.path.isfile(p):
            h.update(f.encode())
            with open(p, "rb") as fh:
                h.update(fh.read())
    h.update(" ".join(ARCH + FLAGS[:4]).encode())
    return h.hexdigest()[:16]


# the files each kernel's code comes from (a recorded profile stays valid while they are unchanged)
KERNEL_SOURCES = {
    "verify": ("sv_kernel.cu", "sv_math.cuh", "sv_ptx.cuh", "sv_internal.h", "sv_small.cu",
               "sv_small.h"),
    "rows": ("sv_rows.cu", "sv_rows.h", "sv_math.cuh", "sv_ptx.cuh", "sv_internal.h"),
    "lmhead": ("sv_lmhead.cu", "sv_lmhead.h", "sv_tc.cuh", "sv_math.cuh", "sv_ptx.cuh"),
    "greedy": ("sv_greedy.cu", "sv_greedy.h", "sv_math.cuh", "sv_ptx.cuh"),
    "small": ("sv_small.cu", "sv_small.h", "sv_math.cuh", "sv_ptx.cuh"),
    "hverify": ("sv_hverify.cu", "sv_hverify.h", "sv_lmhead.cu", "sv_lmhead.h", "sv_tc.cuh",
                "sv_math.cuh", "sv_ptx.cuh"),
}


def kernel_digest(kernel: str) -> str:
    """Hash of the sources one kernel is compiled from, plus the code-generation flags."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        h.update(f.encode())
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(ARCH + FLAGS[:4]).encode())
    return h.hexdigest()[:16]


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile the library if its sources changed (or ``force``); returns the .so path."""
    os.makedirs(OUT_DIR, exist_ok=True)
    stamp = os.path.join(OUT_DIR, "digest.txt")
    digest = source_digest() + ":" + " ".join(extra_flags)
    if not force and os.path.exists(lib_path()) and os.path.exists(stamp):
        with open(stamp) as fh:
            if fh.read().strip() == digest:
                return lib_path()
    exe = nvcc()
    objs = []

    def compile_one(src):
        obj = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        cmd = [exe, *ARCH, *FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path() + ".tmp"
    cmd = [exe, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path())
    with open(stamp, "w") as fh:
        fh.write(digest)
    return lib_path()


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
