"""Compile libgqa_attn.so for sm_103a, in-tree, with nvcc.

The translation units compile in parallel to objects under ``_build/`` and
link into ``libgqa_attn.so`` beside this file. The CUDA runtime is linked
statically; the driver's tensor-map encoder is looked up at run time, so
the library needs no libcuda at link time.

The debug variant ``libgqa_attn_debug.so`` (``-DGQA_DEBUG``, objects under
``_build/debug/``) has every kernel check each computed TMA coordinate and
global index against its tensor's extent; a failed check skips the access
and sets a status bit that ``gqa_attn_get_error`` reports as
GQA_ERR_BOUNDS. The binding loads it instead of the release library when
the environment variable GQA_ATTN_DEBUG is set to 1.

    python -m causal_gqa_attention_flash_gb300.build [-v] [-f] [--debug | --all]
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libgqa_attn.so")
LIB_DEBUG = os.path.join(HERE, "libgqa_attn_debug.so")
SOURCES = ["api.cu", "fwd.cu", "bwd.cu", "bwd_dq.cu", "decode.cu", "noalloc.cu", "rope.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
          "-Xptxas", "-warn-spills", "-I", os.path.join(os.path.dirname(HERE), "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def _stale(obj: str, deps) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def _start(debug: bool, verbose: bool, force: bool, extra_flags):
    """Start the stale compiles of one variant; returns (lib path, objects, [(source, process)])."""
    build_dir = os.path.join(BUILD, "debug") if debug else BUILD
    lib = LIB_DEBUG if debug else LIB
    os.makedirs(build_dir, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    inc = os.path.join(os.path.dirname(HERE), "include")
    headers += [os.path.join(inc, f) for f in os.listdir(inc) if f.endswith(".h")]
    exe = nvcc()
    flags = [*CFLAGS, *(["-DGQA_DEBUG"] if debug else []), *extra_flags]
    procs, objs = [], []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [path, *headers, __file__]):
            cmd = [exe, *ARCH, *flags, "-c", path, "-o", obj]
            if verbose:
                print(" ".join(cmd), flush=True)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    return lib, objs, procs


def _finish(lib, objs, procs, verbose: bool, force: bool):
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode != 0:
            sys.stdout.write(out)
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed on {failed}")
    if force or procs or _stale(lib, objs):
        cmd = [nvcc(), *ARCH, "-shared", "-o", lib, *objs]
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.check_call(cmd)
    return lib


def build_library(verbose: bool = False, force: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Build the release library (or, with debug=True, the checking variant); returns its path."""
    lib, objs, procs = _start(debug, verbose, force, extra_flags)
    return _finish(lib, objs, procs, verbose, force)


def build_all(verbose: bool = False, force: bool = False):
    """Build the release and the debug library, all translation units compiling at once."""
    jobs = [_start(d, verbose, force, ()) for d in (False, True)]
    return [_finish(*j, verbose, force) for j in jobs]


if __name__ == "__main__":
    v, f = "-v" in sys.argv, "-f" in sys.argv
    if "--all" in sys.argv:
        print("\n".join(build_all(verbose=v, force=f)))
    else:
        print(build_library(verbose=v, force=f, debug="--debug" in sys.argv))
