"""Build libpkv.so (sm_103a) from csrc/ with nvcc: one object per translation unit,
compiled in parallel, then linked against the shared CUDA runtime.

With the environment variable PKV_NVTX=1 at build time, every C entry point is wrapped
in an NVTX range named after it (for profiler timelines)."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpkv.so")
SOURCES = ("api.cu", "append.cu", "decode.cu", "prefill.cu", "prefill_tc.cu", "noalloc.cu",
           "graph.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "-I", INCLUDE, "-I", CSRC]


def _defines() -> list:
    return ["-DPKV_NVTX"] if os.environ.get("PKV_NVTX") == "1" else []


def cuda_home() -> str:
    for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if c and os.path.exists(os.path.join(c, "bin", "nvcc")):
            return c
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    raise RuntimeError("nvcc not found: set CUDA_HOME")


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, defines=(), lib: str = LIB,
          obj: str = OBJ) -> str:
    """Compile and link the library; returns its path.  ``defines``, ``lib``, ``obj``:
    extra preprocessor definitions and where a variant build (tests) puts its library and
    objects."""
    home = cuda_home()
    nvcc = os.path.join(home, "bin", "nvcc")
    OBJ_, LIB_ = obj, lib
    os.makedirs(OBJ_, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))]
    headers.append(os.path.join(INCLUDE, "pkv.h"))
    # objects built with other defines are stale
    stamp = os.path.join(OBJ_, "defines.txt")
    defs = _defines() + list(defines)
    want = " ".join(defs)
    if not os.path.exists(stamp) or open(stamp).read() != want:
        force = True
        with open(stamp, "w") as f:
            f.write(want)

    def compile_one(src):
        s = os.path.join(CSRC, src)
        o = os.path.join(OBJ_, src.replace(".cu", ".o"))
        if force or _stale(o, [s, *headers]):
            cmd = [nvcc, *ARCH, *FLAGS, *defs, "-c", s, "-o", o + ".tmp"]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
            if verbose and (r.stdout or r.stderr):
                print(r.stdout, r.stderr, file=sys.stderr)
            os.replace(o + ".tmp", o)
        return o

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    if force or _stale(LIB_, objs):
        libdir = os.path.join(home, "lib64")
        tmp = LIB_ + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
               "-Xlinker", f"-rpath,{libdir}", *(["-ldl"] if _defines() else [])]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB_)
    return LIB_


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
