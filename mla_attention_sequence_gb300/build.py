"""Builds liblaga_mla.so (the C-ABI library) in-tree with nvcc for sm_103a.

    python -m mla_attention_sequence_gb300.build [-v]

Each .cu file under csrc/ compiles to an object in _build/ (in parallel);
the objects link into _build/liblaga_mla.so against the shared CUDA runtime.
Rebuilds only what changed (sources and headers are compared by mtime).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
# LAGA_BUILD_TRACE=1 builds a separate debug library with in-kernel event
# tracing compiled in (see LAGA_TRACE in csrc/ptx.cuh).
TRACE = os.environ.get("LAGA_BUILD_TRACE", "") == "1"
BUILD = os.path.join(HERE, "_build_trace" if TRACE else "_build")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB = os.path.join(BUILD, "liblaga_mla.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def cuda_home() -> str:
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc())))


def _flags(ptxas_verbose: bool):
    f = ["-O3", "-std=c++17", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC", f"-I{INCLUDE}",
         "--expt-relaxed-constexpr", "-Xcompiler", "-Wno-unused-function"]
    if ptxas_verbose:
        f += ["-Xptxas", "-v"]
    if TRACE:
        f += ["-DLAGA_TRACE", f"-DLAGA_TRACE_BY={int(os.environ.get('LAGA_TRACE_BY', '0'))}"]
    return f


def _stale(obj: str, src: str, headers) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(x) > t for x in [src, *headers])


def build(verbose: bool = False, force: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    cc = nvcc()
    jobs = []
    objs = []
    for s in srcs:
        o = os.path.join(BUILD, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        if force or _stale(o, s, headers):
            jobs.append([cc, *_flags(verbose), "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for cmd, r in ex.map(run, jobs):
                if verbose or r.returncode != 0:
                    sys.stderr.write(r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError(f"nvcc failed: {' '.join(cmd)}")
    if jobs or not os.path.exists(LIB):
        link = [cc, *ARCH, "-shared", "-cudart", "shared", "-o", LIB, *objs,
                "-Xlinker", f"-rpath,{os.path.join(cuda_home(), 'lib64')}"]
        r = subprocess.run(link, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link of liblaga_mla.so failed")
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
