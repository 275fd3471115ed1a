"""In-tree build of libuvu.so: host C++ with g++, device code with nvcc for sm_103a only.

The library links the CUDA runtime statically and NVRTC dynamically; it does not link the driver
library, so it loads on machines without a GPU (where only the host-side planner can run).
Objects and the library go to ``_build/`` next to this file.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libuvu.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def cuda_home() -> str:
    for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if c and os.path.exists(os.path.join(c, "bin", "nvcc")):
            return c
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    raise RuntimeError("CUDA toolkit (nvcc) not found")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith((".cpp", ".cu")))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".h")]
    hs.append(os.path.join(ROOT, "include", "uvu.h"))
    return hs


def _stale(target, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    cuda = cuda_home()
    inc = ["-I", os.path.join(ROOT, "include"), "-I", CSRC, "-I", os.path.join(cuda, "include")]
    os.makedirs(OUT, exist_ok=True)
    srcs = _sources()
    hdrs = _headers()
    jobs = []
    objs = []
    for s in srcs:
        o = os.path.join(OUT, os.path.basename(s) + ".o")
        objs.append(o)
        if not force and not _stale(o, [s] + hdrs):
            continue
        if s.endswith(".cu"):
            cmd = [os.path.join(cuda, "bin", "nvcc"), *ARCH, "-lineinfo", "-O3", "-std=c++17",
                   "-Xcompiler", "-fPIC", *inc, "-c", s, "-o", o]
        else:
            cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-Wno-unused-function", *inc,
                   "-c", s, "-o", o]
        jobs.append(cmd)

    def run(cmd):
        if verbose:
            print(" ".join(cmd))
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"build failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, max(1, len(jobs)))) as ex:
        for msg in ex.map(run, jobs):
            if verbose and msg:
                print(msg)
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        run([os.path.join(cuda, "bin", "nvcc"), *ARCH, "-shared", *objs, "-o", tmp,
             "-L", os.path.join(cuda, "lib64"), "-lnvrtc", "-cudart", "static",
             "-Xlinker", "-rpath," + os.path.join(cuda, "lib64")])
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
