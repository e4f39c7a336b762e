"""Build libigemm.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

The translation units compile in parallel into ``_build/`` and link into
``libigemm.so`` next to this file, with the CUDA runtime linked statically so
that loading the library needs no GPU (only the kernels do).
"""

from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libigemm.so")
SOURCES = ["api.cu", "prep.cu", "gemm_i4i4.cu", "gemm_small.cu", "gemm_w4a8.cu", "gemm_fp8.cu", "gemm_bs.cu", "host.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _compile(src: str, ptxas_verbose: bool) -> tuple[str, str]:
    obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), "-c", "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC,
           os.path.join(CSRC, src), "-o", obj]
    if ptxas_verbose:
        cmd.insert(2, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stdout + r.stderr


def _newest_source_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "igemm.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def up_to_date() -> bool:
    return os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= _newest_source_mtime()


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = True) -> str:
    if not force and up_to_date() and not ptxas_verbose:
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    import fcntl
    # one builder at a time (the ranks of one job, parallel test workers): the
    # others wait here and find the library up to date
    with open(os.path.join(BUILD_DIR, ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        if not force and up_to_date() and not ptxas_verbose:
            return LIB_PATH
        return _build_locked(ptxas_verbose, quiet)


def _build_locked(ptxas_verbose: bool, quiet: bool) -> str:
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, ptxas_verbose), SOURCES))
    logs = "".join(log for _, log in results)
    if ptxas_verbose or not quiet:
        sys.stderr.write(logs)
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc(), "-shared", *ARCH, "-cudart", "static", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    build(force=True, ptxas_verbose="-v" in sys.argv, quiet=False)
    print(LIB_PATH)
