"""In-tree build of libtra.so for sm_103a (nvcc, one -gencode, translation units in parallel).

The check build (libtra_check.so, -DTRA_CHECK) is the same library with a bounds test before
every plain global access of the CUDA-core kernels and the tensor-core warp stores; the binding
loads it instead when the environment sets TRA_CHECK=1."""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB = os.path.join(HERE, "libtra.so")
LIB_CHECK = os.path.join(HERE, "libtra_check.so")
BUILD_DIR = os.path.join(os.path.dirname(HERE), "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtra.so")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))


def headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".h")]
    return hs + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]


def stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in sources() + headers() + [__file__])


def build(force: bool = False, verbose: bool = False, check: bool = False, both: bool = False) -> str:
    """Compile every CUDA/C++ source under csrc/ and link libtra.so next to this file
    (check=True: libtra_check.so with -DTRA_CHECK; both=True: both libraries, all translation
    units compiled in one parallel pass).  Returns the (first) library's path."""
    variants = [False, True] if both else [check]
    todo = [v for v in variants if force or stale(LIB_CHECK if v else LIB)]
    if not todo:
        return LIB_CHECK if (check and not both) else LIB
    nvcc = _nvcc()

    def compile_one(job):
        src, chk = job
        bdir = BUILD_DIR + ("_check" if chk else "")
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *(["-DTRA_CHECK"] if chk else []), "-c", src, "-o", obj]
        if src.endswith(".cpp"):
            cmd[1:1] = ["-x", "cu"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    srcs = sources()
    for v in todo:
        os.makedirs(BUILD_DIR + ("_check" if v else ""), exist_ok=True)
    jobs = [(s, v) for v in todo for s in srcs]
    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 8))) as ex:
        objs = list(ex.map(compile_one, jobs))
    for v in todo:
        lib = LIB_CHECK if v else LIB
        tmp = lib + ".tmp"
        mine = [o for o, (_, c) in zip(objs, jobs) if c == v]
        # the driver API (tensor-map encoding) is reached through the runtime's entry-point query
        r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *mine], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB_CHECK if (check and not both) else LIB
