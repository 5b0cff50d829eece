"""In-tree build of libspx.so (sm_103a) with nvcc and the host C++ compiler.

Translation units compile in parallel; the link uses nvcc with the static CUDA
runtime.  Nothing here is imported by the compute path.
"""
from __future__ import annotations

import glob
import hashlib
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ = os.path.join(PKG, "_obj")
LIB = os.path.join(PKG, "libspx.so")
# the bounds-checked build: the same sources with -DSPX_CHECK (every index a kernel
# reads from the caller's arrays is tested before use; see csrc/spx_check.cuh)
OBJ_CHECK = os.path.join(PKG, "_obj_check")
LIB_CHECK = os.path.join(PKG, "libspx_check.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _cuda_home() -> str:
    return os.path.dirname(os.path.dirname(os.path.realpath(_nvcc())))


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _deps():
    return sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                  glob.glob(os.path.join(INCLUDE, "*.h")))


def _compile_cmd(src: str, obj: str, extra=()):
    inc = ["-I", INCLUDE, "-I", CSRC, "-I", os.path.join(_cuda_home(), "include")]
    if src.endswith(".cu"):
        return [_nvcc(), *ARCH, "-lineinfo", "-O3", "-std=c++17", "--expt-relaxed-constexpr",
                "-Xcompiler", "-fPIC,-ffp-contract=off", *inc, *extra, "-c", src, "-o", obj]
    return ["g++", "-O2", "-std=c++17", "-fPIC", "-ffp-contract=off", "-fno-fast-math", *inc, *extra,
            "-c", src, "-o", obj]


def _stamp(src: str, extra) -> str:
    h = hashlib.sha1()
    for p in [src, *_deps()]:
        h.update(open(p, "rb").read())
    h.update(" ".join(_compile_cmd(src, "x", extra)).encode())
    return h.hexdigest()[:16]


def build(force: bool = False, verbose: bool = False, extra=(), checked: bool = False) -> str:
    """Compile every translation unit (in parallel) and link libspx.so (checked=True: libspx_check.so)."""
    obj_dir, lib = (OBJ_CHECK, LIB_CHECK) if checked else (OBJ, LIB)
    if checked:
        extra = (*extra, "-DSPX_CHECK")
    os.makedirs(obj_dir, exist_ok=True)
    jobs = []
    objs = []
    for src in _sources():
        base = os.path.splitext(os.path.basename(src))[0]
        obj = os.path.join(obj_dir, f"{base}.{_stamp(src, extra)}.o")
        objs.append(obj)
        if force or not os.path.exists(obj):
            jobs.append((src, obj))

    def run(job):
        src, obj = job
        cmd = _compile_cmd(src, obj + ".tmp", extra)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(obj + ".tmp", obj)
        return r.stderr if verbose else ""

    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for out in ex.map(run, jobs):
                if out:
                    print(out)
    exports = os.path.join(CSRC, "libspx.map")  # the exported symbols: the C ABI only
    newest = max([os.path.getmtime(o) for o in objs] + [os.path.getmtime(exports)])
    if force or jobs or not os.path.exists(lib) or os.path.getmtime(lib) < newest:
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-Xcompiler", "-fPIC", "-Xlinker",
               f"--version-script={exports}"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
        keep = set(objs)
        for o in glob.glob(os.path.join(obj_dir, "*.o")):
            if o not in keep:
                os.remove(o)
    return lib


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checked="--checked" in sys.argv))
