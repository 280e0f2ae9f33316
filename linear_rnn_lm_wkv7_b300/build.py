"""Build libwkv7.so in-tree with nvcc for sm_103a (B300).

    python linear_rnn_lm_wkv7_b300/build.py [--force] [-v] [--debug]

(Run it by path: importing the package itself loads libwkv7.so, which this script makes.)

Each source compiles to an object under _build/ (in parallel), then one link makes the shared library.
nvcc cross-compiles without a GPU.  The shared library links the CUDA runtime dynamically so that it
shares one runtime instance with PyTorch.

--debug makes libwkv7_debug.so with device-side bounds checks (WKV7_DEBUG_CHECKS): an access outside
its buffer is skipped and recorded in the library's debug status word instead of being made (see
wkv7_debug_status() in include/wkv7.h).  The binding loads it when WKV7_LIBRARY names it.
"""
from __future__ import annotations

import concurrent.futures
import hashlib
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libwkv7.so")
LIB_DEBUG = os.path.join(PKG, "libwkv7_debug.so")
SOURCES = ["wkv7_api.cu", "wkv7_fwd.cu", "wkv7_fwdc.cu", "wkv7_chain.cu", "wkv7_bwd.cu", "wkv7_bwd2.cu",
           "wkv7_colmat.cu", "wkv7_xop.cu", "wkv7_decode.cu", "wkv7_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
FLAGS = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return hs + [os.path.join(INCLUDE, "wkv7.h")]


def _newest(paths) -> float:
    return max(os.path.getmtime(p) for p in paths)


def _compile(src: str, obj: str, flags, verbose: bool):
    cmd = [NVCC, *flags, "-c", src, "-o", obj + ".tmp"]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n" + res.stdout + res.stderr)
    os.replace(obj + ".tmp", obj)
    return res.stderr


def build(force: bool = False, verbose: bool = False, debug: bool = False, defines=(), out: str | None = None) -> str:
    """Compile every source for sm_103a and link the library; returns its path.  `defines` adds -D flags
    (e.g. a different default for a tuning constant) into a library at `out`."""
    lib = out or (LIB_DEBUG if debug else LIB)
    flags = list(FLAGS) + (["-DWKV7_DEBUG_CHECKS=1"] if debug else []) + [f"-D{d}" for d in defines]
    tag = hashlib.sha1(" ".join(flags).encode()).hexdigest()[:10]
    objdir = os.path.join(ROOT, "_build", tag)
    os.makedirs(objdir, exist_ok=True)
    hdr_time = _newest(_headers())
    jobs = []
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(objdir, s.replace(".cu", ".o"))
        if force or not os.path.exists(obj) or os.path.getmtime(obj) < max(os.path.getmtime(src), hdr_time):
            jobs.append((src, obj))
    objs = [os.path.join(objdir, s.replace(".cu", ".o")) for s in SOURCES]
    if jobs:
        with concurrent.futures.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            logs = list(ex.map(lambda j: _compile(j[0], j[1], flags, verbose), jobs))
        if verbose:
            sys.stderr.write("".join(logs))
    if jobs or force or not os.path.exists(lib) or os.path.getmtime(lib) < _newest(objs):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [NVCC, *ARCH, "-shared", "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64",
               "-o", tmp] + objs
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc link failed:\n" + res.stdout + res.stderr)
        os.replace(tmp, lib)
    return lib


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    return os.path.getmtime(LIB) < _newest([os.path.join(CSRC, s) for s in SOURCES] + _headers())


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
