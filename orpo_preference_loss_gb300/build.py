"""Build liborpo_head.so in-tree with nvcc for sm_103a (GB300).

Each .cu file is compiled in parallel into an object, then linked into a shared
library against the shared CUDA runtime (the one PyTorch also loads).  The
result lives in ``orpo_preference_loss_gb300/_build/`` (git-ignored).  A build
is skipped when the library is newer than every source and header.

``build(debug=True)`` makes the bounds-checked variant ``liborpo_head_debug.so``
in ``_build_debug/``: the same sources with ORPO_DEBUG_BOUNDS, where every
computed index is checked against its buffer and a miss is reported in the
status word (ORPO_STATUS_BOUNDS) instead of touching memory.
"""

from __future__ import annotations

import fcntl
import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB_NAME = "liborpo_head.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)
DEBUG_OUT_DIR = os.path.join(PKG, "_build_debug")
DEBUG_LIB_PATH = os.path.join(DEBUG_OUT_DIR, "liborpo_head_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-O2", "-Xptxas", "-v"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found; the CUDA toolkit is required to build liborpo_head")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(ROOT, "include", "*.h")) + [os.path.abspath(__file__)])


def up_to_date(debug: bool = False) -> bool:
    lib = DEBUG_LIB_PATH if debug else LIB_PATH
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile the library if needed; returns the path of the shared object.

    Safe to call from several processes at once (ranks of one job): a file lock lets one of them
    build while the others wait and then find the library up to date."""
    lib, out = (DEBUG_LIB_PATH, DEBUG_OUT_DIR) if debug else (LIB_PATH, OUT_DIR)
    if not force and up_to_date(debug):
        return lib
    os.makedirs(out, exist_ok=True)
    with open(os.path.join(out, ".build.lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        try:
            if not force and up_to_date(debug):
                return lib
            return _build_locked(verbose, debug)
        finally:
            fcntl.flock(lock, fcntl.LOCK_UN)


def _build_locked(verbose: bool, debug: bool) -> str:
    nvcc = nvcc_path()
    srcs = _sources()
    lib, out = (DEBUG_LIB_PATH, DEBUG_OUT_DIR) if debug else (LIB_PATH, OUT_DIR)
    flags = NVCC_FLAGS + (["-DORPO_DEBUG_BOUNDS"] if debug else [])
    objs = [os.path.join(out, os.path.basename(s)[:-3] + ".o") for s in srcs]

    def compile_one(pair):
        src, obj = pair
        cmd = [nvcc, *ARCH, *flags, "-I", os.path.join(ROOT, "include"), "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, r

    with ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(compile_one, zip(srcs, objs)))
    failed = False
    for src, r in results:
        if r.returncode != 0:
            failed = True
            sys.stderr.write(f"--- nvcc failed on {src}\n{r.stdout}\n{r.stderr}\n")
        elif verbose:
            sys.stderr.write(f"--- {os.path.basename(src)}\n{r.stderr}")
    if failed:
        raise RuntimeError("liborpo_head build failed")
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"liborpo_head link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
