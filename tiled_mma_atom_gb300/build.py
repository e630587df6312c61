"""Build libtmg.so in-tree from csrc/*.cu with nvcc for sm_103a.

Each translation unit compiles in parallel; the objects link into one shared
library with the CUDA runtime linked statically.  Nothing here needs a GPU.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libtmg.so")
# the debug build: every store of D and every access to split-K scratch in
# the kernels checked against its buffer (-DTMG_DEBUG_BOUNDS)
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "libtmg_debug.so")
SOURCES = ["api.cu", "ffma.cu", "tc_bf16.cu", "tc2_bf16.cu", "tc2_fused.cu", "skinny.cu", "mxfp4.cu",
           "mxfp4_pair.cu", "pack.cu", "w4a8.cu", "w4a8_skinny.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-Wall",
                "-I", CSRC, "-I", INCLUDE]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found")
    return path


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "tmg.h"))
    files.append(os.path.abspath(__file__))
    return files


def stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _deps())


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None,
          debug_bounds: bool = False) -> str:
    lib, bdir = (LIB_DEBUG, BUILD_DEBUG) if debug_bounds else (LIB, BUILD)
    if not force and not stale(lib):
        return lib
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    extra = (extra or []) + (["-DTMG_DEBUG_BOUNDS"] if debug_bounds else [])

    def compile_one(src: str) -> str:
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        cmd = [cc] + FLAGS + extra + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def _code_only(text: str) -> str:
    """C++ source without its comments and blank lines: what the compiler
    sees, so that editing a comment does not disown a profile."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = []
    for line in text.splitlines():
        # drop a // comment unless the // sits inside a string literal
        cut = line.find("//")
        if cut >= 0 and line.count('"', 0, cut) % 2 == 0:
            line = line[:cut]
        line = line.rstrip()
        if line:
            out.append(line)
    return "\n".join(out)


def source_hash(name) -> str:
    """sha256 of the code (comments stripped) of csrc/<name> (a file name or a
    list of them) plus the shared device header: identifies the kernel a
    profile was taken from."""
    import hashlib
    h = hashlib.sha256()
    names = [name] if isinstance(name, str) else list(name)
    for f in names + ["device.cuh"]:
        p = os.path.join(CSRC, f)
        if os.path.exists(p):
            with open(p, encoding="utf-8") as fh:
                h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


if __name__ == "__main__":
    v = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None
    print(build(force=True, verbose=v or bool(extra), extra=extra, debug_bounds="--debug-bounds" in sys.argv))
