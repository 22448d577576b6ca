"""Builds libhs.so (the C-ABI library) in-tree for sm_103a with nvcc.

Each .cu file under csrc/ is compiled to an object in parallel, then linked
into one shared library next to this file.  The CUDA runtime is linked
statically, so the library only needs the driver at run time.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libhs.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

SOURCES = ["hs_api.cu", "hs_append.cu", "hs_score.cu", "hs_select.cu", "hs_attention.cu", "hs_attention_mla.cu",
           "hs_static.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libhs.so")


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "hs.h"), __file__]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, trace: bool | None = None) -> str:
    """Compile and link if anything changed; returns the library path.  trace=True
    (default: environment variable HS_WITH_TRACE=1) compiles the per-CTA phase
    timeline in, for performance work; the library then writes it to the file
    named by HS_TRACE_OUT when a handle is destroyed."""
    if trace is None:
        trace = os.environ.get("HS_WITH_TRACE") == "1"
    flags_file = os.path.join(BUILD, "flags.txt")
    flags = "trace" if trace else "release"
    built_flags = open(flags_file).read() if os.path.exists(flags_file) else ""
    if (not force and built_flags == flags and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= _deps_mtime()):
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if trace:
        extra.append("-DHS_WITH_TRACE")

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *CFLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for _, err in results:
            if err:
                print(err, file=sys.stderr)
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(flags_file, "w") as f:
        f.write(flags)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv, trace=True if "--trace" in sys.argv else None)
    print(LIB)
