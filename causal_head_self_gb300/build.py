"""Build libattn_sm103a.so in-tree: nvcc for sm_103a, one object per
translation unit (compiled in parallel), linked with nvcc -shared.
The CUDA runtime is linked statically; the driver is reached at run time
through cudaGetDriverEntryPointByVersion, so the library loads on a machine
without a GPU driver (it then fails at the first call)."""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libattn_sm103a.so")
# the checked variant (-DATTN_CHECK): every kernel range-checks the copies it
# issues and reports a failed check as ATTN_ERR_CHECK instead of issuing it
BUILD_CHECK = os.path.join(PKG, "_build_check")
LIB_CHECK = os.path.join(PKG, "libattn_sm103a_check.so")
SOURCES = ["attn_api.cu", "prefill_sm103a.cu", "decode_sm103a.cu", "backward_sm103a.cu"]
HEADERS = ["sm103a_ptx.cuh", "prefill_sm103a.cuh", "prefill_k64_sm103a.cuh", "decode_sm103a.cuh",
           "decode_tc_sm103a.cuh", "backward_sm103a.cuh", "backward256_sm103a.cuh", "launch.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build the library")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, check: bool = False) -> str:
    """Compile the library (or, with check=True, its range-checked variant)
    and return its path."""
    nvcc = _nvcc()
    build_dir, lib_path = (BUILD_CHECK, LIB_CHECK) if check else (BUILD, LIB)
    flags = FLAGS + (["-DATTN_CHECK"] if check else [])
    os.makedirs(build_dir, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in HEADERS] + [
        os.path.join(os.path.dirname(PKG), "include", "attn.h")]
    objs, jobs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + headers):
            jobs.append([nvcc, *ARCH, *flags, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stdout.write(r.stdout + r.stderr)

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        list(ex.map(run, jobs))
    if jobs or force or _stale(lib_path, objs):
        tmp = lib_path + f".tmp{os.getpid()}"
        run([nvcc, *ARCH, "-shared", "-o", tmp, *objs])
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, check="--check" in sys.argv))
