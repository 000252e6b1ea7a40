"""Build libvc.so (the C-ABI library) in-tree for sm_103a with nvcc.

Each .cu under csrc/ is compiled by nvcc and each .cpp (host-only code, the
scheduler) by the host C++ compiler, in parallel, to object files that are
then linked into lossless_compressed_kv_gb300/libvc.so.  Run as a script
(python lossless_compressed_kv_gb300/build.py): importing the package needs
the library this builds.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libvc.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
CXX = os.environ.get("CXX", "g++")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    os.makedirs(OBJ, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu"))) + sorted(glob.glob(os.path.join(CSRC, "*.cpp")))
    hdrs = sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [os.path.join(ROOT, "include", "vc.h")]
    objs = []
    jobs = []
    for s in srcs:
        base, ext = os.path.splitext(os.path.basename(s))
        o = os.path.join(OBJ, base + (".o" if ext == ".cu" else ".host.o"))
        objs.append(o)
        if force or _stale(o, [s] + hdrs):
            if ext == ".cu":
                jobs.append([NVCC, *ARCH, *FLAGS, *extra, "-c", s, "-o", o])
            else:
                jobs.append([CXX, "-O2", "-std=c++17", "-fPIC", "-fvisibility=hidden", "-I",
                             os.path.join(ROOT, "include"), "-I", CSRC, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode:
            raise RuntimeError("nvcc failed: " + " ".join(cmd))

    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        list(ex.map(run, jobs))
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + ".tmp%d" % os.getpid()
        run([NVCC, *ARCH, "-shared", "-o", tmp, *objs])
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
