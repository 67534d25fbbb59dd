"""Builds libqmm.so for sm_103a, in-tree, with nvcc.

Each .cu file under csrc/ compiles to an object in parallel; the objects link
into ``lib/libqmm.so``.  The CUDA runtime is linked statically and the driver
API (tensor-map encoding) is reached through cudaGetDriverEntryPointByVersion,
so the library needs no link against libcuda.

    python -m bit_weight_quantized_gb300.build [-v]
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys
import sysconfig
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIBDIR = os.path.join(HERE, "lib")
LIB = os.path.join(LIBDIR, "libqmm.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers_digest() -> str:
    h = hashlib.sha1()
    for d in (CSRC, INCLUDE):
        for f in sorted(os.listdir(d)):
            if f.endswith((".h", ".cuh")):
                with open(os.path.join(d, f), "rb") as fh:
                    h.update(f.encode() + fh.read())
    return h.hexdigest()


def _compile(src: str, verbose: bool, ptxas_verbose: bool) -> str:
    obj = os.path.join(BUILD, src[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
    if ptxas_verbose:
        cmd += ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
    if verbose and (res.stdout or res.stderr):
        sys.stderr.write(res.stdout + res.stderr)
    return obj


def build(verbose: bool = False, force: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile every kernel and link lib/libqmm.so; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    stamp = os.path.join(BUILD, "headers.sha1")
    digest = _headers_digest()
    old = open(stamp).read() if os.path.exists(stamp) else ""
    stale_headers = force or old != digest
    todo = []
    for src in _sources():
        obj = os.path.join(BUILD, src[:-3] + ".o")
        if stale_headers or not os.path.exists(obj) or \
                os.path.getmtime(obj) < os.path.getmtime(os.path.join(CSRC, src)):
            todo.append(src)
    if todo:
        with cf.ThreadPoolExecutor(max_workers=min(8, len(todo))) as ex:
            list(ex.map(lambda s: _compile(s, verbose, ptxas_verbose), todo))
    objs = [os.path.join(BUILD, s[:-3] + ".o") for s in _sources()]
    if todo or not os.path.exists(LIB):
        tmp = LIB + f".{os.getpid()}.tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, LIB)
    with open(stamp, "w") as fh:
        fh.write(digest)
    build_fastcall(verbose)
    return LIB


FAST_SRC = os.path.join(CSRC, "pyfast.c")


def fastcall_path() -> str:
    """Where the fast-call extension (csrc/pyfast.c) is built."""
    return os.path.join(LIBDIR, "_qmmfast" + (sysconfig.get_config_var("EXT_SUFFIX") or ".so"))


def build_fastcall(verbose: bool = False) -> Optional[str]:
    """Compiles the CPython fast-call extension with the host C compiler.  It is
    optional: without Python's headers (or a compiler) the binding keeps
    calling through ctypes, so a failure here only warns."""
    out = fastcall_path()
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(FAST_SRC):
        return out
    inc = sysconfig.get_paths().get("include", "")
    cc = os.environ.get("CC") or shutil.which("gcc") or shutil.which("cc")
    if not cc or not os.path.exists(os.path.join(inc, "Python.h")):
        sys.stderr.write("note: fast-call extension not built (no C compiler or Python.h)\n")
        return None
    tmp = out + f".{os.getpid()}.tmp"
    cmd = [cc, "-O2", "-shared", "-fPIC", "-I", inc, FAST_SRC, "-o", tmp]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        sys.stderr.write(f"note: fast-call extension not built:\n{res.stderr}\n")
        return None
    if verbose and res.stderr:
        sys.stderr.write(res.stderr)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    v = "-v" in sys.argv
    print(build(verbose=v, force="-f" in sys.argv, ptxas_verbose=v))
