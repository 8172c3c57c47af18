"""Builds libspconv.so in-tree for sm_103a (GB300) with nvcc.

The translation units (the kernel instances, one per output-channels-per-warp
count, the launcher and the host library) compile in parallel and link against
the shared CUDA runtime, so the library and PyTorch share one runtime and one
primary context.

build(debug=True) builds the bounds-checked variant, libspconv_debug.so (the
same sources with -DSPCONV_DEBUG=1, objects in _build_debug/): every kernel
access is checked against its extent first and a failed check sets bit 2 of
the device error word instead of touching memory.  Point the Python binding
at it with SPCONV_LIBRARY=<path>.

build(trace=True) builds libspconv_trace.so (-DSPCONV_TRACE=1, objects in
_build_trace/): every forward block records its start, first-stage-ready and
pipeline-end times, read back with spconv_trace_read (bench.py --timeline).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libspconv.so")
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "libspconv_debug.so")
BUILD_TRACE = os.path.join(HERE, "_build_trace")
LIB_TRACE = os.path.join(HERE, "libspconv_trace.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["spconv_fwd.cu", "spconv_fwd_q1.cu", "spconv_fwd_q2.cu", "spconv_fwd_q4.cu",
           "spconv_fwd_q8.cu", "spconv_fwd_pairs.cu", "spconv_fwd_plane.cu", "spconv_fwd_cols.cu",
           "spconv_fwd_colpair.cu", "spconv_fwd_colpair5.cu", "spconv_fwd_tight.cu",
           "spconv_ws.cu", "spconv_io.cu", "spconv_noalloc.cu", "spconv_host.cpp"]
HEADERS = [os.path.join(CSRC, "spconv_internal.h"), os.path.join(CSRC, "spconv_kernel.cuh"),
           os.path.join(ROOT, "include", "spconv.h")]


def cuda_home() -> str:
    env = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if env:
        return env
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _nvcc() -> str:
    return os.path.join(cuda_home(), "bin", "nvcc")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False,
          trace: bool = False) -> str:
    if debug and trace:
        raise ValueError("the bounds-checked and trace builds are separate libraries")
    bdir, lib_path = ((BUILD_DEBUG, LIB_DEBUG) if debug else
                      (BUILD_TRACE, LIB_TRACE) if trace else (BUILD, LIB))
    os.makedirs(bdir, exist_ok=True)
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", *ARCH, "-lineinfo", "-I", os.path.join(ROOT, "include"),
              "-Xcompiler", "-fPIC,-fvisibility=hidden,-O3,-Wall", *extra_flags]
    if debug:
        common.append("-DSPCONV_DEBUG=1")
    if trace:
        common.append("-DSPCONV_TRACE=1")
    objs, procs = [], []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(bdir, src + ".o")
        objs.append(obj)
        if force or _stale(obj, [path, *HEADERS]):
            cmd = [nvcc, *common, "-c", path, "-o", obj]
            if src.endswith(".cu"):
                cmd[1:1] = ["-Xptxas", "-v"] if verbose else []
            procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT, text=True)))
    for cmd, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode:
            sys.stderr.write(out)
        if p.returncode:
            raise RuntimeError("nvcc failed: " + " ".join(cmd))
    if force or procs or _stale(lib_path, objs):
        rpath = os.path.join(cuda_home(), "lib64")
        cmd = [nvcc, "-shared", *ARCH, "-o", lib_path + ".tmp", *objs, "-cudart", "shared",
               "-Xlinker", "-rpath," + rpath]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link failed: " + " ".join(cmd))
        os.replace(lib_path + ".tmp", lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                debug="--debug" in sys.argv, trace="--trace" in sys.argv))
