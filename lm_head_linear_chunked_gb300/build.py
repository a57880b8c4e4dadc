"""Builds liblce.so, the library behind include/lce.h, in-tree for sm_103a,
and its bounds-checking twin liblce_debug.so (the same sources compiled with
LCE_DEBUG: every kernel checks its computed indices and TMA store
coordinates and reports a failed check as LCE_ERR_BOUNDS).

Each .cu file is compiled separately (in parallel) with nvcc and linked
into one shared library with the CUDA runtime linked statically, so that
loading it needs no GPU and no driver (the driver is only touched when a
function enqueues work).
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
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "liblce.so")
LIB_DEBUG = os.path.join(PKG, "liblce_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", CSRC, "-I", INCLUDE]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    return files + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)] + [__file__]


def _variant(debug: bool):
    """(library path, object folder, extra nvcc flags) of the release or the bounds-checking build."""
    if debug:
        return LIB_DEBUG, BUILD_DIR + "_debug", ["-DLCE_DEBUG"]
    return LIB, BUILD_DIR, []


def up_to_date(debug: bool = False) -> bool:
    lib = _variant(debug)[0]
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def _compile(nvcc: str, src: str, obj_dir: str, flags: list[str], verbose: bool) -> str:
    obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc, *ARCH, *flags, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or r.returncode:
        sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}")
    return obj


def _link(nvcc: str, lib: str, objs: list[str]) -> None:
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode:
        sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        raise RuntimeError(f"link of {os.path.basename(lib)} failed")
    os.replace(tmp, lib)


def build(force: bool = False, verbose: bool = False, debug: bool = False, both: bool = False) -> str:
    """Builds the release library (or, with debug, the bounds-checking one;
    with both, the two together in one pool of compiler processes) unless it
    is newer than every source.  Returns the path of the (release) library."""
    variants = [False, True] if both else [debug]
    todo = [v for v in variants if force or not up_to_date(v)]
    if todo:
        nvcc = _nvcc()
        jobs = []
        for v in todo:
            lib, obj_dir, extra = _variant(v)
            os.makedirs(obj_dir, exist_ok=True)
            jobs += [(v, src, obj_dir, NVCC_FLAGS + extra) for src in sources()]
        with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            objs = list(ex.map(lambda j: (j[0], _compile(nvcc, j[1], j[2], j[3], verbose)), jobs))
        for v in todo:
            _link(nvcc, _variant(v)[0], [o for w, o in objs if w == v])
    return _variant(debug and not both)[0]


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv,
                both="--both" in sys.argv))
