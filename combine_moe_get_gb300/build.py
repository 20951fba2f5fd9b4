"""Build ``libmoe_get.so`` in place: nvcc for sm_103a, one object per .cu
(compiled in parallel), linked against the shared CUDA runtime so that the
library and PyTorch share one runtime instance in a process."""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmoe_get.so")
# the same library compiled with MOE_PROFILE: every kernel warp records its start and end (moe_trace_enable)
TRACE_LIB = os.path.join(HERE, "libmoe_get_trace.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe_get.so")


def _cuda_lib_dirs(nvcc: str) -> list[str]:
    root = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    dirs = [os.path.join(root, "lib64")] + glob.glob(os.path.join(root, "targets", "*", "lib"))
    return [d for d in dirs if os.path.isdir(d)]


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False, defines: tuple = (), lib: str = LIB,
          build_dir: str = BUILD_DIR) -> str:
    """Compile and link the library in place. `defines` (e.g. ("MOE_TUNE_X=4",))
    builds a variant with other compile-time settings; the default build has none."""
    if not force and up_to_date(lib):
        return lib
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)
    common = [nvcc, *ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              "-I", INCLUDE, "--expt-relaxed-constexpr", *(f"-D{d}" for d in defines)]

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = common + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    link = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs]
    for d in _cuda_lib_dirs(nvcc):
        link += ["-Xlinker", f"-rpath,{d}"]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build_trace(force: bool = False, verbose: bool = False) -> str:
    """libmoe_get_trace.so: the library compiled with MOE_PROFILE (per-warp timer records)."""
    return build(force, verbose, defines=("MOE_PROFILE=1",), lib=TRACE_LIB, build_dir=BUILD_DIR + "_trace")


if __name__ == "__main__":
    print(build(force=True, verbose=True))
